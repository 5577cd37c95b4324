"""Planted mistakes in the oracle must each fail at least one pin.

The oracle source has build-time switches (ORACLE_MUTANT=n) that plant one
plausible mistake each; this test compiles every variant on the CPU and checks
that the pin set rejects it, so that the pins are known to be able to catch
the kind of error they guard against.
"""
import pytest

from oracle import Oracle
from tests import oracle_pins as P

MUTANTS = {
    1: "softmax scale dropped",
    2: "wrong sign in the exponent",
    3: "wrong query-head -> kv-head map",
    4: "causal diagonal key dropped",
    5: "V rows read as K",
    6: "wrong in-page offset",
    7: "log-sum-exp in base 2",
    8: "merge drops the second term",
    9: "cache write to the wrong slot",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_pins_catch_planted_mistake(mutant):
    orc = Oracle(mutant)
    failed = []
    for pin in P.ALL_PINS:
        try:
            ok, _ = pin(orc)
        except Exception:  # an error raised by the mutant counts as caught
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {mutant} ({MUTANTS[mutant]})"

"""Planted mistakes in the oracle must each fail at least one pin.

The oracle source has build-time switches (ORACLE_MUTANT=n) that plant one
plausible mistake each; this test compiles every variant on the CPU and checks
that the pin set rejects it, so that the pins are known to be able to catch
the kind of error they guard against.  Mistakes 1-9, 16 and 17 are in the
attention, merge, cascade and cache-write oracle (checked against the pin set
of oracle_pins.py), 10-15 in its fp8 e4m3 functions (checked against the fp8
pins of test_oracle_fp8.py).
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
    16: "cascade suffix starts one key late",
    17: "cascade prefix pass stops one key early",
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


FP8_MUTANTS = {
    10: "e4m3 ties not to the even code",
    11: "e4m3 no saturation above 448",
    12: "scale multiplies instead of divides",
    13: "e4m3 subnormals off by a factor 2",
    14: "K and V scales swapped on dequantisation",
    15: "e4m3 exponent bias 8",
}


def _fp8_pins():
    from tests import test_oracle_fp8 as F

    return [
        ("worked encodings", F.test_worked_encodings),
        ("every finite code", F.test_values_and_round_trip_of_every_finite_code),
        ("scale divides", F.test_scale_divides_before_rounding),
        ("bf16 equivalence", lambda o: F.test_fp8_attention_equals_bf16_attention_on_the_dequantised_pool(o, 0.5, 0.25)),
        ("cache write", F.test_fp8_cache_write_is_the_quantised_row),
        ("dense softmax", lambda o: F.test_fp8_attention_equals_dense_softmax_with_any_scale(o, 0.0371, 0.0173)),
    ]


@pytest.mark.parametrize("mutant", sorted(FP8_MUTANTS), ids=lambda m: FP8_MUTANTS[m].replace(" ", "_"))
def test_fp8_pins_catch_planted_mistake(mutant):
    orc = Oracle(mutant)
    failed = []
    for name, pin in _fp8_pins():
        try:
            pin(orc)
        except Exception:  # an assertion (or an error raised by the mutant) counts as caught
            failed.append(name)
    assert failed, f"no fp8 pin caught mutant {mutant} ({FP8_MUTANTS[mutant]})"


def test_fp8_pins_pass_on_the_oracle():
    orc = Oracle(0)
    for name, pin in _fp8_pins():
        pin(orc)

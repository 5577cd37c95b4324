"""The fp64 oracle against its pins (CPU only)."""
import pytest

from tests import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle, pin):
    ok, detail = pin(oracle)
    assert ok, detail

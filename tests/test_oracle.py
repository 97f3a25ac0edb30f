"""The fp64 oracle against its pins (closed forms, invariants, library routines,
finite differences and hand-worked fixtures).  CPU only."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin, orc):
    pin(orc)

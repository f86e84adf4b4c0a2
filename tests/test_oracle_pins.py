"""The oracle against facts the definitions fix (closed forms, invariants,
library special cases, finite differences).  CPU only."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)

"""The CPU oracle against its pins (closed forms, invariants, the pages' L = 4
table, library float conversions).  CPU only."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()

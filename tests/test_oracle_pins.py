"""The CPU oracle against its pins (no GPU): see tests/oracle_pins.py."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.PINS, ids=[p.__name__ for p in P.PINS])
def test_pin(pin):
    pin()

"""The float64 oracle against what the pages and the mathematics fix.

CPU only.  Each pin is described in tests/oracle_pins.py.
"""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(orc, pin):
    pin(orc)

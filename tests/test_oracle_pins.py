"""The oracle against its pins (worked examples, closed forms, library
routines, invariants).  CPU only."""
import pytest

import oracle as O
from oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def L():
    return O.lib()


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin, L):
    pin(L)

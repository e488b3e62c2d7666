"""The CPU oracle against its pins (closed forms, invariants, brute force, library routines, page values)."""
import pytest

import oracle_pins
from oracle import Oracle


@pytest.fixture(scope="module")
def o():
    return Oracle()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)

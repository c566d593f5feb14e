"""The fp64 oracle against closed forms, invariants and an unpaged brute force."""
import pytest

import pins
from oracle import oracle as orc


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(orc.load())

"""The f64 oracle against hand-worked fixtures, closed forms, invariants and PyTorch f64."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()

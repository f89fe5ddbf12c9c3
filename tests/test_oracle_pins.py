"""The CPU oracle against closed forms, invariants, library routines, brute
force and hand-worked fixtures (no GPU)."""
import pytest

import oracle.kvmem as ora
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(ora)

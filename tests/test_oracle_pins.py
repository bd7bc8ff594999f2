"""The CPU oracle against the pins (no GPU)."""
import pytest

import oracle.attention as orc
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(orc)

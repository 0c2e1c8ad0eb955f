"""The CPU oracle against its pins (no GPU needed)."""
import pytest

import oracle as O
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(O.lib())

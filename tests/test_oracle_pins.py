"""The CPU oracle against its pins (golden values, closed forms, invariants,
library special cases, brute force).  No GPU."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)

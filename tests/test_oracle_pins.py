"""The fp64 oracle against what the pages and mathematics fix (CPU only)."""

import pytest

from oracle import recurrence
from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(recurrence._load())

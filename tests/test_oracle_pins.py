"""The oracle against what the pages and mathematics fix (CPU only)."""
import pytest

from oracle import q4_oracle as O
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(O)

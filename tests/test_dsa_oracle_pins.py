"""The DSA indexer oracle against its pins (CPU)."""
import pytest

from dsa_oracle_pins import PINS
from oracle import dsa


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_dsa_oracle_pin(pin):
    pin(dsa.load())

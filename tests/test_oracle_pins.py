"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle_pins
from oracle import oracle


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)

"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def L():
    return oracle.lib()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS + oracle_pins.CHECK_PINS, ids=lambda p: p.__name__)
def test_pin(pin, L):
    pin(L)

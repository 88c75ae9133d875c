"""The oracle against its pins (CPU only)."""

import pytest

import oracle.mqa as oracle_mqa

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(oracle_mqa)

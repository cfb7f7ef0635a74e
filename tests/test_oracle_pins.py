"""The oracle against its pins (library routines, closed forms, invariants)."""

import pytest

from oracle import kda_oracle as ko

import oracle_pins as pins


@pytest.fixture(scope="module")
def oracle():
    return ko.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=[p.__name__ for p in pins.ALL_PINS])
def test_pin(pin, oracle):
    pin(oracle)

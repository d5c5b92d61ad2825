"""The CPU oracle against its pins (library routines, closed forms, invariants)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.lib()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__[4:])
def test_oracle_pin(lib, pin):
    oracle_pins.run_pin(pin, lib)

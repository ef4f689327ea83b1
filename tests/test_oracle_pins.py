"""The CPU oracle against facts fixed by the pages and by the mathematics
(closed forms, invariants, a textbook float64 routine, brute force)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)

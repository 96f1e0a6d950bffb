"""The FP64 oracle against the pages' printed values and closed forms (CPU only)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(oracle, pin):
    pin(oracle)


def test_oracle_threads(oracle):
    assert oracle.num_threads() >= 1

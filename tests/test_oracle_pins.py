"""The oracle against what the pages and mathematics fix (no GPU)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL, ids=[p.__name__ for p in pins.ALL])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)

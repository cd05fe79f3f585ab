"""The oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    if pin is oracle_pins.pin_brute_force_tiny:
        pytest.importorskip("mpmath")
    pin(oracle_lib)

"""The CPU oracle against facts the attention pages and mathematics fix (no GPU)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    if pin is oracle_pins.pin_bruteforce_tiny:
        pytest.importorskip("mpmath")
    pin(oracle.default())

"""The float64 oracle against facts the KDA pages and mathematics fix (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("name", list(oracle_pins.PINS))
def test_pin(name):
    fn, bar = oracle_pins.PINS[name]
    val = float(fn())
    assert val <= bar, f"{name}: violation {val:.3e} > {bar:.0e}"

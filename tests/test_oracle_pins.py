"""The oracle against its pins (CPU only).

See ``oracle_pins.py`` for what each pin checks and what fixes it.
"""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS,
                         ids=[p.__name__ for p in oracle_pins.ALL_PINS])
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)

"""The oracle against closed forms, invariants, brute force and golden points."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("pin", oracle_pins.PREOP_PINS, ids=lambda f: f.__name__)
def test_preop_pin(orc, pin):
    pin(orc)

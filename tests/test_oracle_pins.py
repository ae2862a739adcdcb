"""The oracle against its pins (closed forms, library routines, brute force,
the verifier example of dflash_engine.py, and the model card's invariants)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()

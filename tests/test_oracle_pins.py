"""The oracle against the pages' worked examples, closed forms, library
reductions and brute force (see ``oracle_pins.py``). CPU only."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__[4:])
def test_pin(oracle, pin):
    pin(oracle)

"""The FP64 oracle against its pins (closed forms, invariants, library special
cases, chunked-WY algebra).  CPU only."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())

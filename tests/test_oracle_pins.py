"""The oracle against its pins (hand-worked cases, library routines, invariants, a dense second
formulation).  CPU only."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())

"""The oracle against closed forms, invariants, library routines and brute
force (CPU only).  See tests/oracle_pins.py for what each check pins."""
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.forward)

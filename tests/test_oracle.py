"""Pins of the fp64 oracle (CPU only): see tests/oracle_pins.py for what each check pins."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.default())

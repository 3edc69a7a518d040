"""Pins of the fp64 oracle (CPU only)."""
import pytest

import oracle
from oracle_pin_checks import ALL_CHECKS


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle.default())

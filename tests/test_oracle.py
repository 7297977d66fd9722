"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", oracle_pins.CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(lib, check):
    check(lib)

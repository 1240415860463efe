"""The CPU oracle against its pins (no GPU). See ``oracle_pins.py``."""

import pytest

import oracle
from oracle_pins import ALL_CHECKS


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library()


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__[6:])
def test_oracle_pin(check, lib):
    check(lib)

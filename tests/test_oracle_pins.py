"""The CPU oracle against its pins (closed forms, special cases, brute force)."""

import pytest

import oracle.whitematter as O
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(O)

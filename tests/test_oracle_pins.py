"""The oracle against its pins (closed forms, invariants, brute force); CPU only."""

import pytest

import oracle_checks


@pytest.mark.parametrize("check", oracle_checks.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, check):
    check(orc)

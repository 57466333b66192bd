"""The CPU oracle against its pins (no GPU).  See oracle_checks.py."""
import pytest

import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()


def test_rounding_helpers():
    oc.check_rounding_helpers()

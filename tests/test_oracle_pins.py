"""The oracle against its pins (CPU only). See tests/oracle_checks.py."""
import pytest

import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(olib, check):
    check(olib)

"""The fp64 oracle against facts fixed outside it (CPU only)."""
import pytest

import oracle
from tests import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle.asp_oracle)

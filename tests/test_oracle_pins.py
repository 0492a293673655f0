"""The fp64 oracle against hand-derived values, closed forms, invariants and
library routines (CPU only)."""

import pytest

import oracle.block_hybrid as ob
from tests import oracle_checks


@pytest.mark.parametrize("check", oracle_checks.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(ob)

"""The float64 oracle against facts other than itself (library special
cases, closed forms, invariants). CPU only."""

import pytest

import oracle.paged_attention as orc
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS,
                         ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(orc)

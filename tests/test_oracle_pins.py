"""The CPU oracle against its pins (see tests/oracle_pins.py for what pins what)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=[c.__name__ for c in P.ALL_CHECKS])
def test_oracle_pin(orc, check):
    check(orc)

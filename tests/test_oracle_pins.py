"""The CPU oracle against its pins (library routines, brute force, closed
forms, error bounds and hand-worked examples).  CPU only."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle.default())

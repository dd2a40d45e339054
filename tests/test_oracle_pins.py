"""The CPU oracle against closed forms, invariants, torch and exact arithmetic."""
import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__[len("check_"):])
def test_oracle_pin(check, oracle_lib):
    check(oracle_lib)

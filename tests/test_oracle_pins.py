"""The CPU oracle against its pins (no GPU)."""
import pytest

from tests import oracle_pin_checks as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check()

"""The CPU oracle against its pins (see tests/oracle_pins.py)."""
import pytest

from oracle import moe_oracle

from . import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(moe_oracle)

"""The CPU oracle against facts that do not come from the oracle itself."""
import pytest

from tests import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check, oracle_lib):
    check(oracle_lib)

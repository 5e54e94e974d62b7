"""The CPU oracle against facts fixed outside itself (no GPU needed)."""
import pytest

import _pins
from oracle import Oracle


@pytest.fixture(scope="module")
def oracle():
    return Oracle()


@pytest.mark.parametrize("check", _pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(oracle, check):
    check(oracle)

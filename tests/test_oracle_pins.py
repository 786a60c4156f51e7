"""The oracle against facts fixed outside it (closed forms, a hand-worked example,
finite differences, invariants, the composed formulation and torch's SDPA)."""
import pytest

import oracle
from oracle_pins import PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)

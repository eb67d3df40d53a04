"""The CPU oracle against closed forms, library routines and invariants."""

import pytest

import oracle_pins
from oracle import taco_oracle


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(taco_oracle)

"""The oracle against its pins (CPU only)."""

import pytest

import oracle.draft as oracle_draft
import oracle.step as oracle_step
from oracle_pins import ALL_PINS
from oracle_pins_draft import DRAFT_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle_step)


@pytest.mark.parametrize("pin", DRAFT_PINS, ids=lambda p: p.__name__)
def test_draft_oracle_pin(pin):
    pin(oracle_draft)

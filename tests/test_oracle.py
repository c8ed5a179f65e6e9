"""The CPU oracle against its pins (library routines, closed forms, paging invariants)."""
import pytest

from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)

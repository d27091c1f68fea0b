"""The CPU oracle against the pages' worked examples, closed forms, a
library attention routine and the pages' invariants (no GPU needed)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(pin):
    pin()

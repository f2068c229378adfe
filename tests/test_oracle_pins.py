"""The CPU oracle against facts that do not come from itself (tests/oracle_pins.py)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_closed_form_against_empirical_uniform_routing():
    P.pin_closed_form_empirical(seeds=200)

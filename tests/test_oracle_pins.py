"""The CPU oracle against its pins (closed forms, hand-worked values, library special cases,
exact identities and invariants). See ``pins.py`` for what each pin fixes."""

import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, orc_lib):
    pin(orc_lib)

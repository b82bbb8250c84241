"""The CPU oracle checked against what the pages and the mathematics fix
(see tests/_pins.py for the pins and their sources)."""
import pytest

import _pins
import oracle


@pytest.fixture(scope="module")
def lib():
    return oracle.lib()


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(lib, pin):
    pin(lib)

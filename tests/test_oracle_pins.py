"""The shipped CPU oracle against its pins (no GPU)."""

import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)

"""The CPU oracle against facts that do not come from it (see tests/pins.py)."""
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)

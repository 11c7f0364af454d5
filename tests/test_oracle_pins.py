"""The oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import oracle
from _pins import ALL_PINS


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)

"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle
from tests import _pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(lib, pin):
    pin(lib)

"""The fp64 oracle against its pins (tests/pins.py): CPU only."""
import pytest

import oracle
from pins import PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("name", list(PINS))
def test_pin(orc, name):
    PINS[name](orc)

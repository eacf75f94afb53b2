"""The fp64 oracle against its pins (closed forms, invariants, library
special cases, finite differences).  CPU only."""
import pytest

import oracle.attention as att
import oracle.merge as mrg
import oracle.permute as prm
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(att, mrg, prm)

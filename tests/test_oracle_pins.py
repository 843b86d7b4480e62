"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.get())


def test_rejects_bad_arguments():
    o = oracle.get()
    x = np.zeros(12)
    with pytest.raises(ValueError):
        o.forward(x, 1, 4, 3, 3, 0, None, None, 1e-5)   # G does not divide C
    with pytest.raises(ValueError):
        o.forward(x, 1, 4, 3, 0, 0, None, None, 1e-5)   # G = 0
    with pytest.raises(ValueError):
        o.forward(x, 1, 4, 3, 2, 2, None, None, 1e-5)   # unknown layout


def test_empty_extents_are_noops():
    o = oracle.get()
    y, mean, rstd = o.forward(np.zeros(0), 2, 4, 0, 2, 1, None, None, 1e-5)
    assert y.size == 0
    dx, dg, db = o.backward(np.zeros(0), np.zeros(0), 0, 4, 5, 2, 0, None, 1e-5)
    assert dx.size == 0 and np.all(dg == 0) and np.all(db == 0)

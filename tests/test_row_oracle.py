"""The fp64 LayerNorm / RMSNorm oracle against its pins, and a mutation test
showing that every planted mistake is caught (CPU only).

Mutants: unbiased variance, eps outside the square root, gamma indexed by
row, the LayerNorm mean-gradient term dropped, the xhat term's sign flipped,
the mean-gradient term kept for RMSNorm, dgamma of raw x, dbeta weighted by
gamma.
"""
import numpy as np
import pytest

import oracle
from tests import row_pins


@pytest.mark.parametrize("pin", row_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_row_pin(pin):
    pin(oracle.get_row())


def test_row_oracle_rejects_bad_arguments():
    ro = oracle.get_row()
    with pytest.raises(ValueError):
        ro.ln_forward(np.zeros(0), 0, 0, None, None, 1e-5)    # N = 0
    with pytest.raises(ValueError):
        ro.rms_forward(np.zeros(4), 2, 2, None, -1.0)         # negative eps


@pytest.mark.parametrize("mutant", list(range(1, 9)))
def test_every_row_mutant_fails_a_pin(mutant, tmp_path):
    ro = oracle.RowOracle(mutant, outdir=str(tmp_path))
    assert ro.mutant == mutant
    caught = []
    for pin in row_pins.ALL_PINS:
        try:
            pin(ro)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"

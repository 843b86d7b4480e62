"""The GPU parity inputs are discriminating (CPU only, oracle only).

A parity case only proves something if a plausible kernel mistake would miss
its tolerance.  For the cases whose 16-byte vectors span several groups, run
with the correlated dy of tests/cases.py, the oracle copies with one planted
mistake in dx (mean(gamma*dy) term dropped, xhat*mean(gamma*dy*xhat) term
dropped, that term's sign flipped, gamma indexed by group where a group has
several channels) must each give a
dx outside the tolerance the GPU is held to; and neighbouring groups must
have clearly different statistics, so that a kernel applying one group's
coefficients to a neighbour's channels fails too.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from backward_normalization_gb300 import synth
from tests import checks
from tests.cases import SPANNING, strong_dy

DX_MUTANTS = (3, 4, 5, 8)


@pytest.fixture(scope="module")
def mutants(tmp_path_factory):
    d = tmp_path_factory.mktemp("mutants")
    return {k: oracle.Oracle(k, outdir=str(d)) for k in DX_MUTANTS}


def _dx(o, inp, w):
    L = synth.LAYOUTS[w.layout]
    dx, _, _ = o.backward(inp["dy"].double().numpy(), inp["x"].double().numpy(), w.N, w.C, w.HW,
                          w.G, L, inp["gamma"].double().numpy(), w.eps)
    return dx


@pytest.mark.parametrize("name,w", SPANNING, ids=[c[0] for c in SPANNING])
def test_planted_dx_mistakes_miss_the_tolerance(name, w, mutants):
    inp = strong_dy(synth.make_inputs(w, "cpu", seed=0), w)
    ref = _dx(oracle.get(), inp, w)
    # the reference rounded to the storage type passes (the check is attainable)
    checks.assert_out("dx", synth.torch.from_numpy(ref).to(synth.DTYPES[w.dtype]), ref, w.dtype)
    for k, o in mutants.items():
        if k == 8 and w.C == w.G:
            continue  # one channel per group: gamma by group is gamma by channel
        with pytest.raises(AssertionError):
            checks.assert_out(f"dx (mutant {k})", _dx(o, inp, w), ref, w.dtype)


@pytest.mark.parametrize("name,w", SPANNING, ids=[c[0] for c in SPANNING])
def test_neighbouring_groups_differ(name, w):
    """Group means of neighbouring groups differ by more than 0.05 of the
    group's standard deviation in at least 90 % of the pairs, from the
    per-channel offsets.  Using a neighbour's mean moves y = (x - mean)*rstd*
    gamma + beta by that difference times rstd*gamma (gamma ~ 1 here): five
    times the 16-bit atol and 500 times the fp32 bound."""
    inp = synth.make_inputs(w, "cpu", seed=0)
    L = synth.LAYOUTS[w.layout]
    mean, var, rstd = oracle.get().stats(inp["x"].double().numpy(), w.N, w.C, w.HW, w.G, L, w.eps)
    m = mean.reshape(w.N, w.G)
    r = rstd.reshape(w.N, w.G)
    if w.G < 2:
        pytest.skip("one group")
    sep = np.abs(np.diff(m, axis=1)) * r[:, 1:]
    assert np.mean(sep > 0.05) >= 0.9, sep

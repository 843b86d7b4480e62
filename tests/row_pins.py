"""Pins for the fp64 LayerNorm / RMSNorm oracle (``oracle.RowOracle``): checks
against facts fixed by the definitions and by mathematics, independent of the
oracle's own code.

Each ``pin_*`` takes a RowOracle and raises AssertionError when it disagrees.
They run against the real oracle (test_row_oracle.py) and against copies with
one planted mistake each, so that every mistake is shown to be caught.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b) / (1.0 + np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


def _fr(lst):
    return np.array([float(Fraction(v)) for v in lst])


def _case(seed, M, N, offset=0.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(M * N) * 1.3 + offset
    dy = rng.standard_normal(M * N)
    gamma = rng.standard_normal(N)
    beta = rng.standard_normal(N)
    return x, dy, gamma, beta


def pin_row_golden_hand_worked(ro):
    """Hand-derived examples with exact rational answers (tests/golden)."""
    d = json.load(open(os.path.join(GOLDEN, "row_hand_worked.json")))
    L = d["ln"]
    y, mean, rstd = ro.ln_forward(L["x"], L["M"], L["N"], L["gamma"], L["beta"], L["eps"])
    dx, dg, db = ro.ln_backward(L["dy"], L["x"], L["M"], L["N"], L["gamma"], L["eps"])
    for name, got in (("mean", mean), ("rstd", rstd), ("y", y), ("dx", dx), ("dgamma", dg),
                      ("dbeta", db)):
        _close(got, _fr(L[name]), 1e-14, f"ln {name}")
    R = d["rms"]
    y, rstd = ro.rms_forward(R["x"], R["M"], R["N"], R["gamma"], R["eps"])
    dx, dg = ro.rms_backward(R["dy"], R["x"], R["M"], R["N"], R["gamma"], R["eps"])
    for name, got in (("rstd", rstd), ("y", y), ("dx", dx), ("dgamma", dg)):
        _close(got, _fr(R[name]), 1e-14, f"rms {name}")


def pin_ln_is_groupnorm_with_one_group(ro):
    """A LayerNorm row is a GroupNorm sample with one group and HW = 1 (channels
    = features), computed by the separately pinned GroupNorm oracle."""
    gn = oracle.get()
    for seed, (M, N), affine in ((0, (5, 7), True), (1, (3, 16), False), (2, (1, 9), True)):
        x, dy, gamma, beta = _case(seed, M, N, offset=2.5)
        g, b = (gamma, beta) if affine else (None, None)
        eps = 1e-3
        y, mean, rstd = ro.ln_forward(x, M, N, g, b, eps)
        dx, dg, db = ro.ln_backward(dy, x, M, N, g, eps)
        yr, mr, rr = gn.forward(x, M, N, 1, 1, 1, g, b, eps)
        dxr, dgr, dbr = gn.backward(dy, x, M, N, 1, 1, 1, g, eps)
        for name, got, ref in (("y", y, yr), ("mean", mean, mr), ("rstd", rstd, rr), ("dx", dx, dxr),
                               ("dgamma", dg, dgr), ("dbeta", db, dbr)):
            _close(got, ref, 1e-12, f"ln vs groupnorm {name} (seed {seed})")


def pin_ln_invariants(ro):
    """Per row: sum of xhat = 0, mean of xhat^2 = var/(var + eps), and
    sum of dx = 0 for any gamma."""
    M, N, eps = 4, 11, 0.25
    x, dy, gamma, _ = _case(3, M, N, offset=-1.0)
    y, mean, rstd = ro.ln_forward(x, M, N, None, None, eps)  # y = xhat
    xh = y.reshape(M, N)
    var = np.var(x.reshape(M, N), axis=1)
    assert np.max(np.abs(xh.sum(axis=1))) < 1e-12, "sum of xhat"
    _close((xh ** 2).mean(axis=1), var / (var + eps), 1e-12, "mean xhat^2")
    dx, _, _ = ro.ln_backward(dy, x, M, N, gamma, eps)
    assert np.max(np.abs(dx.reshape(M, N).sum(axis=1))) < 1e-12, "sum of dx"


def pin_rms_invariants(ro):
    """With eps = 0: mean of xhat^2 = 1 per row and sum of x*dx = 0 (the
    gradient is orthogonal to the scaling direction)."""
    M, N = 3, 10
    x, dy, gamma, _ = _case(4, M, N, offset=0.7)
    y, rstd = ro.rms_forward(x, M, N, None, 0.0)
    _close((y.reshape(M, N) ** 2).mean(axis=1), np.ones(M), 1e-13, "rms mean xhat^2")
    dx, _ = ro.rms_backward(dy, x, M, N, gamma, 0.0)
    s = (x.reshape(M, N) * dx.reshape(M, N)).sum(axis=1)
    assert np.max(np.abs(s)) < 1e-12, "rms sum of x*dx"


def pin_rms_is_layernorm_on_zero_mean_rows(ro):
    """For rows of zero mean the two norms coincide in y, rstd and dgamma."""
    M, N, eps = 3, 8, 1e-2
    x, dy, gamma, _ = _case(5, M, N)
    x = (x.reshape(M, N) - x.reshape(M, N).mean(axis=1, keepdims=True)).reshape(-1)
    y1, _, r1 = ro.ln_forward(x, M, N, gamma, None, eps)
    y2, r2 = ro.rms_forward(x, M, N, gamma, eps)
    _close(y2, y1, 1e-12, "y")
    _close(r2, r1, 1e-12, "rstd")
    _, dg1, _ = ro.ln_backward(dy, x, M, N, gamma, eps)
    _, dg2 = ro.rms_backward(dy, x, M, N, gamma, eps)
    _close(dg2, dg1, 1e-12, "dgamma")


def _fd(f, v, h=1e-6):
    g = np.zeros_like(v)
    for i in range(v.size):
        a, b = v.copy(), v.copy()
        a[i] += h
        b[i] -= h
        g[i] = (f(a) - f(b)) / (2 * h)
    return g


def pin_ln_finite_differences(ro):
    """dx, dgamma, dbeta are the gradients of L = sum(dy * y)."""
    M, N, eps = 2, 5, 1e-3
    x, dy, gamma, beta = _case(6, M, N, offset=0.3)
    loss = lambda xv, gv, bv: float(np.dot(dy, ro.ln_forward(xv, M, N, gv, bv, eps)[0]))
    dx, dg, db = ro.ln_backward(dy, x, M, N, gamma, eps)
    _close(dx, _fd(lambda v: loss(v, gamma, beta), x), 1e-7, "ln dx")
    _close(dg, _fd(lambda v: loss(x, v, beta), gamma), 1e-7, "ln dgamma")
    _close(db, _fd(lambda v: loss(x, gamma, v), beta), 1e-7, "ln dbeta")


def pin_rms_finite_differences(ro):
    """dx and dgamma are the gradients of L = sum(dy * y)."""
    M, N, eps = 2, 6, 1e-3
    x, dy, gamma, _ = _case(7, M, N, offset=0.4)
    loss = lambda xv, gv: float(np.dot(dy, ro.rms_forward(xv, M, N, gv, eps)[0]))
    dx, dg = ro.rms_backward(dy, x, M, N, gamma, eps)
    _close(dx, _fd(lambda v: loss(v, gamma), x), 1e-7, "rms dx")
    _close(dg, _fd(lambda v: loss(x, v), gamma), 1e-7, "rms dgamma")


def pin_single_feature_rows(ro):
    """N = 1: a LayerNorm row has zero variance, so y = beta and dx = 0;
    RMSNorm of one feature is x / sqrt(x^2 + eps)."""
    M, eps = 4, 1e-2
    x, dy, gamma, beta = _case(8, M, 1)
    y, mean, rstd = ro.ln_forward(x, M, 1, gamma, beta, eps)
    _close(y, np.full(M, beta[0]), 1e-14, "ln y")
    _close(mean, x, 1e-14, "ln mean")
    dx, _, db = ro.ln_backward(dy, x, M, 1, gamma, eps)
    assert np.max(np.abs(dx)) < 1e-14, "ln dx"
    _close(db, [dy.sum()], 1e-14, "ln dbeta")
    y, rstd = ro.rms_forward(x, M, 1, None, eps)
    _close(y, x / np.sqrt(x * x + eps), 1e-14, "rms y")


ALL_PINS = [pin_row_golden_hand_worked, pin_ln_is_groupnorm_with_one_group, pin_ln_invariants,
            pin_rms_invariants, pin_rms_is_layernorm_on_zero_mean_rows,
            pin_ln_finite_differences, pin_rms_finite_differences, pin_single_feature_rows]

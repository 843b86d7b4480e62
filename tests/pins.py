"""Pins for the fp64 oracle: checks against facts fixed by the definition of
GroupNorm and by mathematics, independent of the oracle's own code.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees.  They are run against the real oracle (test_oracle_pins.py)
and against deliberately broken copies (test_oracle_mutants.py), which shows
that every planted mistake is caught by at least one pin.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- utilities
def nchw_to_nhwc(a, N, C, HW):
    """Re-lay a flat NCHW buffer as NHWC (pure data movement)."""
    return np.ascontiguousarray(np.asarray(a).reshape(N, C, HW).transpose(0, 2, 1)).reshape(-1)


def nhwc_to_nchw(a, N, C, HW):
    return np.ascontiguousarray(np.asarray(a).reshape(N, HW, C).transpose(0, 2, 1)).reshape(-1)


def _rand_case(seed, N, C, HW, G, affine=True, offset=0.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(N * C * HW) * 1.7 + offset
    dy = rng.standard_normal(N * C * HW)
    gamma = rng.standard_normal(C) if affine else None
    beta = rng.standard_normal(C) if affine else None
    return x, dy, gamma, beta


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b) / (1.0 + np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


def _fracs(lst):
    return np.array([float(Fraction(v)) for v in lst])


# ---------------------------------------------------------------- the pins
def pin_golden_hand_worked(o):
    """Hand-derived worked examples (tests/golden), in both layouts."""
    for fname in ("hand_worked_g1.json", "hand_worked_g2.json"):
        d = json.load(open(os.path.join(GOLDEN, fname)))
        N, C, HW, G, eps = d["N"], d["C"], d["HW"], d["G"], d["eps"]
        x = np.array(d["x_nchw"], dtype=np.float64)
        dy = np.array(d["dy_nchw"], dtype=np.float64)
        gamma = np.array(d["gamma"], dtype=np.float64)
        beta = np.array(d["beta"], dtype=np.float64)
        for layout in (0, 1):
            xl = x if layout == 0 else nchw_to_nhwc(x, N, C, HW)
            dyl = dy if layout == 0 else nchw_to_nhwc(dy, N, C, HW)
            y, mean, rstd = o.forward(xl, N, C, HW, G, layout, gamma, beta, eps)
            m2, var, r2 = o.stats(xl, N, C, HW, G, layout, eps)
            dx, dg, db = o.backward(dyl, xl, N, C, HW, G, layout, gamma, eps)
            if layout == 1:
                y = nhwc_to_nchw(y, N, C, HW)
                dx = nhwc_to_nchw(dx, N, C, HW)
            _close(mean, _fracs(d["mean"]), 1e-14, f"{fname} mean L{layout}")
            _close(var, _fracs(d["var"]), 1e-14, f"{fname} var L{layout}")
            _close(rstd, _fracs(d["rstd"]), 1e-14, f"{fname} rstd L{layout}")
            _close(y, _fracs(d["y_nchw"]), 1e-14, f"{fname} y L{layout}")
            _close(dx, _fracs(d["dx_nchw"]), 1e-14, f"{fname} dx L{layout}")
            _close(dg, _fracs(d["dgamma"]), 1e-14, f"{fname} dgamma L{layout}")
            _close(db, _fracs(d["dbeta"]), 1e-14, f"{fname} dbeta L{layout}")


def pin_layernorm_g1(o):
    """G = 1 is a LayerNorm over (C, HW) with per-channel affine; brute force
    with numpy's mean and (biased) var."""
    N, C, HW, eps = 3, 4, 5, 1e-3
    x, _, gamma, beta = _rand_case(1, N, C, HW, 1, offset=2.0)
    xs = x.reshape(N, C, HW)
    m = xs.mean(axis=(1, 2), keepdims=True)
    v = xs.var(axis=(1, 2), keepdims=True)
    ref = (xs - m) / np.sqrt(v + eps) * gamma[None, :, None] + beta[None, :, None]
    for layout in (0, 1):
        xl = x if layout == 0 else nchw_to_nhwc(x, N, C, HW)
        y, mean, rstd = o.forward(xl, N, C, HW, 1, layout, gamma, beta, eps)
        if layout == 1:
            y = nhwc_to_nchw(y, N, C, HW)
        _close(y, ref.reshape(-1), 1e-12, f"layernorm y L{layout}")
        _close(mean, m.reshape(-1), 1e-12, "layernorm mean")
        _close(rstd, (1 / np.sqrt(v + eps)).reshape(-1), 1e-12, "layernorm rstd")


def pin_instancenorm_gc(o):
    """G = C is an InstanceNorm: statistics per (n, c)."""
    N, C, HW, eps = 2, 6, 7, 1e-4
    x, _, gamma, beta = _rand_case(2, N, C, HW, C, offset=-1.0)
    xs = x.reshape(N, C, HW)
    m = xs.mean(axis=2, keepdims=True)
    v = xs.var(axis=2, keepdims=True)
    ref = (xs - m) / np.sqrt(v + eps) * gamma[None, :, None] + beta[None, :, None]
    for layout in (0, 1):
        xl = x if layout == 0 else nchw_to_nhwc(x, N, C, HW)
        y, mean, rstd = o.forward(xl, N, C, HW, C, layout, gamma, beta, eps)
        if layout == 1:
            y = nhwc_to_nchw(y, N, C, HW)
        _close(y, ref.reshape(-1), 1e-12, f"instancenorm y L{layout}")
        _close(mean, m.reshape(-1), 1e-12, "instancenorm mean")


def pin_forward_invariants(o):
    """Per group: sum(xhat) = 0 and mean(xhat^2) = var/(var+eps) (= 1 at eps=0)."""
    N, C, HW, G = 2, 8, 9, 4
    Cg = C // G
    x, _, _, _ = _rand_case(3, N, C, HW, G, affine=False, offset=5.0)
    for eps in (0.0, 0.3):
        y, mean, rstd = o.forward(x, N, C, HW, G, 0, None, None, eps)
        _, var, _ = o.stats(x, N, C, HW, G, 0, eps)
        ys = y.reshape(N, G, Cg * HW)
        s1 = ys.sum(axis=2)
        s2 = (ys ** 2).mean(axis=2)
        assert np.max(np.abs(s1)) < 1e-11, f"sum xhat {np.max(np.abs(s1))}"
        _close(s2.reshape(-1), var / (var + eps), 1e-12, f"mean xhat^2 eps={eps}")


def pin_dx_invariants(o):
    """Per group, for any gamma: sum(dx) = 0 and
    sum(dx * xhat) = rstd * sum(g * xhat) * eps / (var + eps)."""
    N, C, HW, G = 2, 6, 5, 3
    Cg = C // G
    for layout in (0, 1):
        x, dy, gamma, _ = _rand_case(4, N, C, HW, G)
        for eps in (0.0, 0.25):
            dx, _, _ = o.backward(dy, x, N, C, HW, G, layout, gamma, eps)
            xhat, _, rstd = o.forward(x, N, C, HW, G, layout, None, None, eps)
            _, var, _ = o.stats(x, N, C, HW, G, layout, eps)
            if layout == 1:
                dx = nhwc_to_nchw(dx, N, C, HW)
                xhat = nhwc_to_nchw(xhat, N, C, HW)
                dyn = nhwc_to_nchw(dy, N, C, HW)
            else:
                dyn = dy
            g = (dyn.reshape(N, C, HW) * gamma[None, :, None]).reshape(N, G, Cg * HW)
            dxs = dx.reshape(N, G, Cg * HW)
            xh = xhat.reshape(N, G, Cg * HW)
            scale = np.max(np.abs(dxs))
            assert np.max(np.abs(dxs.sum(axis=2))) < 1e-11 * (1 + scale), "sum dx"
            lhs = (dxs * xh).sum(axis=2).reshape(-1)
            rhs = rstd * (g * xh).sum(axis=2).reshape(-1) * eps / (var + eps)
            assert np.max(np.abs(lhs - rhs)) < 1e-11 * (1 + scale), f"sum dx*xhat eps={eps}"


def _loss(o, x, dy, N, C, HW, G, layout, gamma, beta, eps):
    y, _, _ = o.forward(x, N, C, HW, G, layout, gamma, beta, eps)
    return float(np.dot(y, dy))


def pin_finite_differences(o):
    """Central differences of L = sum(dy * y) in fp64 against dx, dgamma, dbeta."""
    N, C, HW, G, eps = 2, 4, 3, 2, 1e-2
    h = 1e-6
    for layout in (0, 1):
        x, dy, gamma, beta = _rand_case(5 + layout, N, C, HW, G)
        dx, dg, db = o.backward(dy, x, N, C, HW, G, layout, gamma, eps)
        fd = np.zeros_like(x)
        for i in range(x.size):
            xp = x.copy(); xp[i] += h
            xm = x.copy(); xm[i] -= h
            fd[i] = (_loss(o, xp, dy, N, C, HW, G, layout, gamma, beta, eps)
                     - _loss(o, xm, dy, N, C, HW, G, layout, gamma, beta, eps)) / (2 * h)
        s = np.max(np.abs(fd))
        assert np.max(np.abs(fd - dx)) < 1e-6 * (1 + s), f"fd dx L{layout}"
        fdg = np.zeros(C)
        fdb = np.zeros(C)
        for c in range(C):
            gp = gamma.copy(); gp[c] += h
            gm = gamma.copy(); gm[c] -= h
            fdg[c] = (_loss(o, x, dy, N, C, HW, G, layout, gp, beta, eps)
                      - _loss(o, x, dy, N, C, HW, G, layout, gm, beta, eps)) / (2 * h)
            bp = beta.copy(); bp[c] += h
            bm = beta.copy(); bm[c] -= h
            fdb[c] = (_loss(o, x, dy, N, C, HW, G, layout, gamma, bp, eps)
                      - _loss(o, x, dy, N, C, HW, G, layout, gamma, bm, eps)) / (2 * h)
        assert np.max(np.abs(fdg - dg)) < 1e-6 * (1 + np.max(np.abs(fdg))), f"fd dgamma L{layout}"
        assert np.max(np.abs(fdb - db)) < 1e-6 * (1 + np.max(np.abs(fdb))), f"fd dbeta L{layout}"


def pin_dbeta_closed_form(o):
    """dbeta_c is the plain sum of dy over n and hw (several samples)."""
    N, C, HW, G = 3, 4, 6, 2
    for layout in (0, 1):
        x, dy, gamma, _ = _rand_case(7, N, C, HW, G)
        _, _, db = o.backward(dy, x, N, C, HW, G, layout, gamma, 1e-5)
        dyn = dy if layout == 0 else nhwc_to_nchw(dy, N, C, HW)
        ref = dyn.reshape(N, C, HW).sum(axis=(0, 2))
        _close(db, ref, 1e-13, f"dbeta L{layout}")


def pin_constant_group(o):
    """A constant group has xhat = 0: y = beta, rstd = eps^-1/2 and
    dx = rstd * (g - mean(g))."""
    N, C, HW, G, eps = 1, 4, 3, 2, 0.04
    x = np.full(N * C * HW, 3.25)
    rng = np.random.default_rng(8)
    dy = rng.standard_normal(N * C * HW)
    gamma = rng.standard_normal(C)
    beta = rng.standard_normal(C)
    y, mean, rstd = o.forward(x, N, C, HW, G, 0, gamma, beta, eps)
    _close(y, np.repeat(beta, HW), 1e-14, "constant y")
    _close(rstd, np.full(G, eps ** -0.5), 1e-14, "constant rstd")
    dx, _, _ = o.backward(dy, x, N, C, HW, G, 0, gamma, eps)
    g = (dy.reshape(C, HW) * gamma[:, None]).reshape(G, -1)
    ref = eps ** -0.5 * (g - g.mean(axis=1, keepdims=True))
    _close(dx, ref.reshape(-1), 1e-13, "constant dx")


def pin_sampled_equals_full(o):
    """The sampled entry points agree with the full ones at random offsets."""
    N, C, HW, G, eps = 2, 6, 10, 3, 1e-5
    for layout in (0, 1):
        x, dy, gamma, beta = _rand_case(9, N, C, HW, G)
        y, mean, rstd = o.forward(x, N, C, HW, G, layout, gamma, beta, eps)
        dx, dg, db = o.backward(dy, x, N, C, HW, G, layout, gamma, eps)
        idx = np.random.default_rng(10).integers(0, x.size, 25)
        ya, ma, ra = o.forward_at(x, N, C, HW, G, layout, gamma, beta, eps, idx)
        dxa, dga, dba = o.backward_at(dy, x, N, C, HW, G, layout, gamma, eps, idx)
        _close(ya, y[idx], 1e-15, "y_at")
        _close(dxa, dx[idx], 1e-15, "dx_at")
        _close(dga, dg, 1e-15, "dgamma_at")
        _close(dba, db, 1e-15, "dbeta_at")


ALL_PINS = [
    pin_golden_hand_worked,
    pin_layernorm_g1,
    pin_instancenorm_gc,
    pin_forward_invariants,
    pin_dx_invariants,
    pin_finite_differences,
    pin_dbeta_closed_form,
    pin_constant_group,
    pin_sampled_equals_full,
]

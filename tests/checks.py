"""Shared comparison helpers for the GPU parity tests.

Tolerances (stated once, used everywhere):
  * fp32 outputs (y, dx of fp32 inputs; mean and rstd always), and the fp64
    storage type (computed in fp32, so held to the fp32 rule):
        max |got - ref| / (1 + |ref|)  <= 1e-4
  * fp16 / bf16 outputs (y, dx):  |got - ref| <= 1e-2 + 1e-2 * |ref|
  * dgamma, dbeta:  ||got - ref||_2 / ||ref||_2 <= 1e-3
The reference is always the fp64 oracle, unrounded.
"""
from __future__ import annotations

import numpy as np
import torch

TOL_F32 = 1e-4
TOL_HALF = 1e-2
TOL_PARAM_L2 = 1e-3


def as_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy().reshape(-1)
    return np.asarray(t, dtype=np.float64).reshape(-1)


def max_rel_f32(got, ref) -> float:
    g, r = as_np(got), as_np(ref)
    if g.size == 0:
        return 0.0
    return float(np.max(np.abs(g - r) / (1.0 + np.abs(r))))


def assert_out(name, got, ref, dtype: str):
    """y or dx: the fp32 rule for fp32 and fp64 data, atol = rtol = 1e-2 otherwise."""
    g, r = as_np(got), as_np(ref)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    if dtype in ("f32", "f64"):
        e = max_rel_f32(g, r)
        assert e <= TOL_F32, f"{name}: max rel err {e:.3e} > {TOL_F32}"
    else:
        bad = np.abs(g - r) > TOL_HALF + TOL_HALF * np.abs(r)
        if np.any(bad):
            i = int(np.argmax(bad))
            raise AssertionError(f"{name}: {int(bad.sum())} elements outside atol=rtol=1e-2, "
                                 f"first at {i}: got {g[i]!r} ref {r[i]!r}")


def assert_stat(name, got, ref):
    e = max_rel_f32(got, ref)
    assert e <= TOL_F32, f"{name}: max rel err {e:.3e} > {TOL_F32}"


def rel_l2(got, ref) -> float:
    g, r = as_np(got), as_np(ref)
    den = np.linalg.norm(r)
    return float(np.linalg.norm(g - r) / (den if den > 0 else 1.0))


def assert_param(name, got, ref):
    e = rel_l2(got, ref)
    assert e <= TOL_PARAM_L2, f"{name}: rel L2 {e:.3e} > {TOL_PARAM_L2}"

"""Shared comparison helpers for the GPU parity tests.

Tolerances (stated once, used everywhere):
  * fp32 outputs (y, dx of fp32 inputs; mean and rstd always), and the fp64
    storage type (computed in fp32, so held to the fp32 rule):
        max |got - ref| / (1 + |ref|)  <= 1e-4
  * fp16 / bf16 outputs (y, dx):  |got - ref| <= 1e-2 + 1e-2 * |ref|
  * dgamma, dbeta:  ||got - ref||_2 / ||ref||_2 <= 1e-3
  * y, dx over a whole tensor, in addition (assert_out_l2):
        ||got - ref||_2 / ||ref||_2 <= u + 1e-4
    with u the unit roundoff of the storage type (2^-8 bf16, 2^-11 fp16,
    2^-24 fp32): rounding each value to nearest moves it by at most u times
    its magnitude, so the rounding alone is within u in relative L2, and
    1e-4 covers the fp32 arithmetic before it.  This catches errors that stay
    under the elementwise absolute floor of 1e-2 when the outputs are small.
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


UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -24, "f64": 2.0 ** -24}


def assert_out_l2(name, got, ref, dtype: str):
    """Relative L2 error of a whole output against the rounding bound."""
    e = rel_l2(got, ref)
    bound = UNIT_ROUNDOFF[dtype] + 1e-4
    assert e <= bound, f"{name}: rel L2 {e:.3e} > {bound:.3e}"
    return e


def assert_param(name, got, ref):
    e = rel_l2(got, ref)
    assert e <= TOL_PARAM_L2, f"{name}: rel L2 {e:.3e} > {TOL_PARAM_L2}"

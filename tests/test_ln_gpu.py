"""GPU parity of the row-normalization kernels (include/ln.h): LayerNorm and
RMSNorm forward/backward through the C ABI against the fp64 row oracle.

Small cases are compared element by element; they cover the vector path (team
widths from 2 to 256 threads), the scalar path (rows whose byte length is not a
multiple of 16, unaligned pointers), M = 1 and N = 1, and the output masks.
The benchmark table's shapes run at full size with y/dx checked on sampled rows
and dgamma/dbeta in full (the oracle takes the rows in blocks).  Tolerances
are those of tests/checks.py.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from backward_normalization_gb300 import gn, synth
from tests import checks

pytestmark = pytest.mark.gpu

RW = synth.RowWorkload

SMALL = [
    RW("ln_f16_32x512", "ln", "f16", 32, 512),
    RW("ln_f16_96x768", "ln", "f16", 96, 768),
    RW("ln_bf16_192x1024", "ln", "bf16", 192, 1024),
    RW("ln_f32_64x4096", "ln", "f32", 64, 4096),
    RW("ln_bf16_40x4096", "ln", "bf16", 40, 4096),
    RW("ln_f16_1000x64", "ln", "f16", 1000, 64),
    RW("ln_f32_300x8", "ln", "f32", 300, 8),
    RW("ln_f16_5x37_scalar", "ln", "f16", 5, 37),
    RW("ln_f32_9x1", "ln", "f32", 9, 1),
    RW("ln_bf16_1x1024", "ln", "bf16", 1, 1024),
    RW("rms_f16_96x768", "rms", "f16", 96, 768),
    RW("rms_bf16_40x4096", "rms", "bf16", 40, 4096),
    RW("rms_f32_64x4096", "rms", "f32", 64, 4096),
    RW("rms_f16_1000x64", "rms", "f16", 1000, 64),
    RW("rms_f32_7x33_scalar", "rms", "f32", 7, 33),
    RW("rms_f16_1x2", "rms", "f16", 1, 2),
]


def _oracle(inp, w, gamma=True, beta=True):
    ro = oracle.get_row()
    x = inp["x"].double().cpu().numpy()
    dy = inp["dy"].double().cpu().numpy()
    g = inp["gamma"].double().cpu().numpy() if gamma else None
    b = inp["beta"].double().cpu().numpy() if beta else None
    if w.op == "ln":
        y, mean, rstd = ro.ln_forward(x, w.M, w.N, g, b, w.eps)
        dx, dg, db = ro.ln_backward(dy, x, w.M, w.N, g, w.eps)
        return dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)
    y, rstd = ro.rms_forward(x, w.M, w.N, g, w.eps)
    dx, dg = ro.rms_backward(dy, x, w.M, w.N, g, w.eps)
    return dict(y=y, rstd=rstd, dx=dx, dgamma=dg)


def _gpu(inp, w, gamma=True, beta=True, want=(True, True)):
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    g = inp["gamma"].cuda() if gamma else None
    b = inp["beta"].cuda() if beta else None
    if w.op == "ln":
        y, mean, rstd = gn.ln_forward(x, w.M, w.N, g, b, w.eps)
        dx, dg, db = gn.ln_backward(dy, x, mean, rstd, w.M, w.N, g, want=want)
        out = dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)
    else:
        y, rstd = gn.rms_forward(x, w.M, w.N, g, w.eps)
        dx, dg = gn.rms_backward(dy, x, rstd, w.M, w.N, g, want_dgamma=want[0])
        out = dict(y=y, rstd=rstd, dx=dx, dgamma=dg)
    torch.cuda.synchronize()
    return out


def _compare(got, ref, w):
    checks.assert_out("y", got["y"], ref["y"], w.dtype)
    checks.assert_out("dx", got["dx"], ref["dx"], w.dtype)
    checks.assert_stat("rstd", got["rstd"], ref["rstd"])
    if "mean" in ref:
        checks.assert_stat("mean", got["mean"], ref["mean"])
    for k in ("dgamma", "dbeta"):
        if got.get(k) is not None and k in ref:
            checks.assert_param(k, got[k], ref[k])


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_row_small_parity(w):
    inp = synth.make_row_inputs(w, "cpu", seed=0)
    _compare(_gpu(inp, w), _oracle(inp, w), w)


# Forward rows longer than a team of 256 threads holds at a small problem's
# 16 values per thread: the plan takes 32 values per thread (LayerNorm then
# stages gamma and beta in shared memory).  The backward's rows stop at 4096.
LONG_FWD = [
    RW("ln_f16_64x8192", "ln", "f16", 64, 8192),
    RW("rms_bf16_3x8192", "rms", "bf16", 3, 8192),
    RW("ln_f32_16x8192", "ln", "f32", 16, 8192),
]


@pytest.mark.parametrize("w", LONG_FWD, ids=[w.name for w in LONG_FWD])
def test_row_forward_long_rows(w):
    inp = synth.make_row_inputs(w, "cpu", seed=5)
    ro = oracle.get_row()
    x = inp["x"].double().numpy()
    g, b = inp["gamma"].double().numpy(), inp["beta"].double().numpy()
    xd, gd, bd = inp["x"].cuda(), inp["gamma"].cuda(), inp["beta"].cuda()
    if w.op == "ln":
        y, mean, rstd = gn.ln_forward(xd, w.M, w.N, gd, bd, w.eps)
        ry, rmean, rrstd = ro.ln_forward(x, w.M, w.N, g, b, w.eps)
        checks.assert_stat("mean", mean, rmean)
    else:
        y, rstd = gn.rms_forward(xd, w.M, w.N, gd, w.eps)
        ry, rrstd = ro.rms_forward(x, w.M, w.N, g, w.eps)
    torch.cuda.synchronize()
    checks.assert_out("y", y, ry, w.dtype)
    checks.assert_stat("rstd", rstd, rrstd)


@pytest.mark.parametrize("w", [SMALL[1], SMALL[3], SMALL[11]], ids=lambda w: w.name)
def test_row_bit_identical_runs(w):
    inp = synth.make_row_inputs(w, "cpu", seed=1)
    a, b = _gpu(inp, w), _gpu(inp, w)
    for k in a:
        if a[k] is None:
            continue
        ta = a[k].view(torch.uint8) if a[k].dtype != torch.float32 else a[k]
        tb = b[k].view(torch.uint8) if b[k].dtype != torch.float32 else b[k]
        assert torch.equal(ta, tb), k


@pytest.mark.parametrize("want", [(True, False), (False, True), (False, False)],
                         ids=["dgamma_only", "dbeta_only", "dx_only"])
def test_row_output_masks(want):
    """Each parameter gradient may be omitted; the others are unchanged."""
    w = SMALL[2]
    inp = synth.make_row_inputs(w, "cpu", seed=2)
    ref = _oracle(inp, w)
    got = _gpu(inp, w, want=want)
    checks.assert_out("dx", got["dx"], ref["dx"], w.dtype)
    assert (got["dgamma"] is not None) == want[0] and (got["dbeta"] is not None) == want[1]
    if want[0]:
        checks.assert_param("dgamma", got["dgamma"], ref["dgamma"])
    if want[1]:
        checks.assert_param("dbeta", got["dbeta"], ref["dbeta"])


@pytest.mark.parametrize("op", ["ln", "rms"])
def test_row_no_affine(op):
    w = RW(f"{op}_f16_64x1024", op, "f16", 64, 1024)
    inp = synth.make_row_inputs(w, "cpu", seed=3)
    _compare(_gpu(inp, w, gamma=False, beta=False), _oracle(inp, w, gamma=False, beta=False), w)


def test_row_misaligned_pointers_and_in_place():
    """Buffers offset by one element take the scalar path; y may overwrite x
    and dx may overwrite dy."""
    w = RW("ln_f16_48x256", "ln", "f16", 48, 256)
    inp = synth.make_row_inputs(w, "cpu", seed=4)
    ref = _oracle(inp, w)
    xb = torch.empty(w.E + 1, dtype=torch.float16, device="cuda")
    x = xb[1:]
    x.copy_(inp["x"])
    dy = inp["dy"].cuda()
    g, b = inp["gamma"].cuda(), inp["beta"].cuda()
    mean = torch.empty(w.M, device="cuda")
    rstd = torch.empty(w.M, device="cuda")
    x_keep = x.clone()
    assert gn.ln_fwd_raw(x, w.M, w.N, g, b, w.eps, x, mean, rstd) == 0  # in place, unaligned
    dg = torch.empty(w.N, device="cuda")
    db = torch.empty(w.N, device="cuda")
    ws = torch.empty(max(gn.ln_workspace_size(w.M, w.N, "f16"), 16), dtype=torch.uint8,
                     device="cuda")
    assert gn.ln_bwd_raw(dy, x_keep, mean, rstd, g, w.M, w.N, dy, dg, db, ws) == 0
    torch.cuda.synchronize()
    checks.assert_out("y", x, ref["y"], w.dtype)
    checks.assert_out("dx", dy, ref["dx"], w.dtype)
    checks.assert_param("dgamma", dg, ref["dgamma"])
    checks.assert_param("dbeta", db, ref["dbeta"])


@pytest.mark.parametrize("op", ["ln", "rms"])
@pytest.mark.parametrize("dtype,N,pads", [("bf16", 1024, (8, 16, 24)), ("f32", 768, (4, 0, 12)),
                                         ("f16", 256, (3, 5, 1))],
                         ids=["bf16_vector", "f32_vector", "f16_scalar_strides"])
def test_row_strided(op, dtype, N, pads):
    """Rows of x, dy and the output lie in wider buffers (ld = N + pad each);
    the results equal the dense computation, and the padding is not touched."""
    M = 37
    w = RW(f"{op}_{dtype}_{M}x{N}", op, dtype, M, N)
    inp = synth.make_row_inputs(w, "cpu", seed=5)
    ref = _oracle(inp, w)
    dt = synth.DTYPES[dtype]
    ldx, ldd, ldo = N + pads[0], N + pads[1], N + pads[2]

    def wide(src, ld):
        b = torch.full((M, ld), 7.0, dtype=dt, device="cuda")
        if src is not None:
            b[:, :N].copy_(src.view(M, N))
        return b

    xb, dyb = wide(inp["x"], ldx), wide(inp["dy"], ldd)
    yb, dxb = wide(None, ldo), wide(None, ldo)
    g, b = inp["gamma"].cuda(), inp["beta"].cuda()
    mean = torch.empty(M, device="cuda")
    rstd = torch.empty(M, device="cuda")
    dg = torch.empty(N, device="cuda")
    db = torch.empty(N, device="cuda")
    ws = torch.empty(max(gn.ln_workspace_size(M, N, dtype), 16), dtype=torch.uint8, device="cuda")
    if op == "ln":
        assert gn.ln_fwd_ex_raw(xb, ldx, M, N, g, b, w.eps, yb, ldo, mean, rstd) == 0
        assert gn.ln_bwd_ex_raw(dyb, ldd, xb, ldx, mean, rstd, g, M, N, dxb, ldo, dg, db, ws) == 0
    else:
        assert gn.rms_fwd_ex_raw(xb, ldx, M, N, g, w.eps, yb, ldo, rstd) == 0
        assert gn.rms_bwd_ex_raw(dyb, ldd, xb, ldx, rstd, g, M, N, dxb, ldo, dg, ws) == 0
    torch.cuda.synchronize()
    checks.assert_out("y", yb[:, :N].reshape(-1), ref["y"], dtype)
    checks.assert_out("dx", dxb[:, :N].reshape(-1), ref["dx"], dtype)
    checks.assert_stat("rstd", rstd, ref["rstd"])
    checks.assert_param("dgamma", dg, ref["dgamma"])
    if op == "ln":
        checks.assert_stat("mean", mean, ref["mean"])
        checks.assert_param("dbeta", db, ref["dbeta"])
    for buf in (yb, dxb):
        assert torch.all(buf[:, N:] == 7.0), "padding written"
    assert gn.ln_fwd_ex_raw(xb, N - 1, M, N, g, b, w.eps, yb, ldo, mean, rstd) == gn.GN_ERR_INVALID


def test_row_empty_and_errors():
    dev = "cuda"
    x = torch.empty(0, device=dev, dtype=torch.float16)
    r = torch.empty(0, device=dev)
    assert gn.ln_fwd_raw(x, 0, 64, None, None, 1e-5, x, r, r) == 0
    dg = torch.full((64,), 3.0, device=dev)
    db = torch.full((64,), 3.0, device=dev)
    assert gn.ln_bwd_raw(x, x, r, r, None, 0, 64, x, dg, db, None) == 0
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(db == 0)
    y = torch.empty(64, device=dev, dtype=torch.float16)
    m = torch.empty(1, device=dev)
    assert gn.ln_fwd_raw(y, 1, 0, None, None, 1e-5, y, m, m) == gn.GN_ERR_INVALID
    assert gn.ln_fwd_raw(y, 1, 64, None, None, -1.0, y, m, m) == gn.GN_ERR_INVALID
    dx = torch.empty_like(y)
    assert gn.ln_bwd_raw(y, y, m, m, None, 1, 64, dx, dg, db, None) == gn.GN_ERR_WORKSPACE


# ------------------------------------------------------------- full sizes
def _sample_rows(M, k=64, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.integers(0, M, k), [0, M - 1]])).astype(np.int64)


@pytest.mark.parametrize("w", synth.ROW_WORKLOADS, ids=[w.name for w in synth.ROW_WORKLOADS])
def test_row_full_size(w):
    """The benchmark table's shapes: y/dx on sampled rows, mean/rstd and
    dgamma/dbeta in full, and a bit-identical rerun."""
    inp = synth.make_row_inputs(w, "cuda", seed=0)
    got = _gpu(inp, w)
    again = _gpu(inp, w)
    for k in got:
        if got[k] is None:
            continue
        ta = got[k].view(torch.uint8) if got[k].dtype != torch.float32 else got[k]
        tb = again[k].view(torch.uint8) if again[k].dtype != torch.float32 else again[k]
        assert torch.equal(ta, tb), k
    del again
    ro = oracle.get_row()
    g = inp["gamma"].double().cpu().numpy()
    b = inp["beta"].double().cpu().numpy()
    rows = _sample_rows(w.M)
    x2 = inp["x"].view(w.M, w.N)
    dy2 = inp["dy"].view(w.M, w.N)
    xs = x2[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    dys = dy2[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    R = rows.size
    if w.op == "ln":
        y, _, _ = ro.ln_forward(xs, R, w.N, g, b, w.eps)
        dx, _, _ = ro.ln_backward(dys, xs, R, w.N, g, w.eps)
    else:
        y, _ = ro.rms_forward(xs, R, w.N, g, w.eps)
        dx, _ = ro.rms_backward(dys, xs, R, w.N, g, w.eps)
    it = torch.from_numpy(rows).cuda()
    checks.assert_out("y", got["y"].view(w.M, w.N)[it], y, w.dtype)
    checks.assert_out("dx", got["dx"].view(w.M, w.N)[it], dx, w.dtype)
    # statistics and parameter gradients over every row, in blocks of rows
    blk = max(1, (1 << 24) // w.N)
    dg = np.zeros(w.N)
    db = np.zeros(w.N)
    mean = np.zeros(w.M)
    rstd = np.zeros(w.M)
    for r0 in range(0, w.M, blk):
        r1 = min(w.M, r0 + blk)
        xb = x2[r0:r1].double().cpu().numpy()
        dyb = dy2[r0:r1].double().cpu().numpy()
        if w.op == "ln":
            _, m, r = ro.ln_forward(xb, r1 - r0, w.N, None, None, w.eps)
            _, dgb, dbb = ro.ln_backward(dyb, xb, r1 - r0, w.N, g, w.eps)
            mean[r0:r1] = m
            db += dbb
        else:
            _, r = ro.rms_forward(xb, r1 - r0, w.N, None, w.eps)
            _, dgb = ro.rms_backward(dyb, xb, r1 - r0, w.N, g, w.eps)
        rstd[r0:r1] = r
        dg += dgb
    checks.assert_stat("rstd", got["rstd"], rstd)
    checks.assert_param("dgamma", got["dgamma"], dg)
    if w.op == "ln":
        checks.assert_stat("mean", got["mean"], mean)
        checks.assert_param("dbeta", got["dbeta"], db)

"""GPU parity of strided views (gn_fwd_ex / gn_bwd_ex) against the fp64 oracle.

Views: channel slices of a wider tensor in both layouts (16-byte aligned and
not), channel planes padded to a pitch, a batch stored channel-major (planes
of one channel for all samples side by side), in-place calls, and backward
calls whose dy, x and dx each have their own strides.  The oracle runs on
dense copies of the same values; every element outside an output view must
keep its sentinel.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from backward_normalization_gb300 import gn, synth
from tests import checks

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


def _view(buf, off, w, s):
    """The [N, C, HW] (NCHW) or [N, HW, C] (NHWC) view of buf at element
    offset off with strides s = (sample, plane or row)."""
    if w.layout == "nchw":
        return buf.as_strided((w.N, w.C, w.HW), (s[0], s[1], 1), off)
    return buf.as_strided((w.N, w.HW, w.C), (s[0], s[1], 1), off)


def _dense(v):
    return v.contiguous().reshape(-1)


def _place(flat, w, total, off, s, dtype):
    """A buffer of `total` elements holding the sentinel everywhere except the
    view, which holds `flat` (given densely in w's layout)."""
    buf = torch.full((total,), SENTINEL, dtype=dtype, device="cuda")
    _view(buf, off, w, s).copy_(flat.view(_view(buf, off, w, s).shape))
    return buf


def _untouched(buf, w, off, s):
    mask = torch.ones_like(buf, dtype=torch.bool)
    _view(mask, off, w, s).fill_(False)
    return bool(torch.all(buf[mask] == SENTINEL))


def _oracle(inp, w):
    o = oracle.get()
    L = synth.LAYOUTS[w.layout]
    x, dy = inp["x"].double().numpy(), inp["dy"].double().numpy()
    g, b = inp["gamma"].double().numpy(), inp["beta"].double().numpy()
    y, mean, rstd = o.forward(x, w.N, w.C, w.HW, w.G, L, g, b, w.eps)
    dx, dg, db = o.backward(dy, x, w.N, w.C, w.HW, w.G, L, g, w.eps)
    return dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)


def _geometry(w, kind):
    """(total elements, offset, strides) of a view of kind `kind`."""
    N, C, HW = w.N, w.C, w.HW
    if kind == "channel_slice":        # channels [k, k + C) of a tensor with C + 2k channels
        k = 8 if w.dtype in ("f16", "bf16") else 4
        Cw = C + 2 * k
        if w.layout == "nchw":
            return N * Cw * HW, k * HW, (Cw * HW, HW)
        return N * HW * Cw, k, (HW * Cw, Cw)
    if kind == "channel_slice_odd":    # the same at an odd offset: the scalar path
        Cw = C + 5
        if w.layout == "nchw":
            return N * Cw * HW + 3, 3 + 2 * HW, (Cw * HW, HW)
        return N * HW * Cw, 3, (HW * Cw, Cw)
    if kind == "padded":               # planes / rows padded to a pitch
        if w.layout == "nchw":
            pitch = HW + 16
            return N * C * pitch, 0, (C * pitch, pitch)
        pitch = C + 16
        return N * HW * pitch, 0, (HW * pitch, pitch)
    if kind == "channel_major":        # planes (rows) of all samples side by side
        if w.layout == "nchw":
            return C * N * HW, 0, (HW, N * HW)
        return HW * N * C, 0, (C, N * C)
    raise ValueError(kind)


CASES = [
    ("fp32_nchw_3x24x20x20_g6", synth.WORKLOADS[0].scaled(name="sv0", N=3, C=24, G=6, H=20, W=20)),
    ("bf16_nhwc_4x64x9x11_g8", synth.WORKLOADS[4].scaled(name="sv4", N=4, C=64, G=8, H=9, W=11)),
    ("fp16_nhwc_2x40x16x16_g4_cg10", synth.WORKLOADS[1].scaled(name="sv1", N=2, C=40, G=4, H=16, W=16)),
    ("fp32_nchw_2x16x64x64_g4_chunks", synth.WORKLOADS[3].scaled(name="sv3", N=2, C=16, G=4, H=64, W=64)),
]
KINDS = ["channel_slice", "channel_slice_odd", "padded", "channel_major"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_strided_views_match_the_oracle(name, w, kind):
    inp = synth.make_inputs(w, "cpu", seed=51)
    ref = _oracle(inp, w)
    dt = synth.DTYPES[w.dtype]
    tot, off, s = _geometry(w, kind)
    # outputs use another geometry than the inputs where there is one
    okind = {"channel_slice": "padded", "padded": "channel_major",
             "channel_major": "channel_slice", "channel_slice_odd": "channel_slice_odd"}[kind]
    otot, ooff, os_ = _geometry(w, okind)
    xb = _place(inp["x"].cuda(), w, tot, off, s, dt)
    dyb = _place(inp["dy"].cuda(), w, otot, ooff, os_, dt)  # dy in a third layout
    yb = torch.full((otot,), SENTINEL, dtype=dt, device="cuda")
    dxb = torch.full((tot,), SENTINEL, dtype=dt, device="cuda")
    gm, bt = inp["gamma"].cuda(), inp["beta"].cuda()
    mean = torch.empty(w.N * w.G, device="cuda")
    rstd = torch.empty(w.N * w.G, device="cuda")
    dg, db = torch.empty(w.C, device="cuda"), torch.empty(w.C, device="cuda")
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, dt)
    x0, y0, dy0, dx0 = xb[off:], yb[ooff:], dyb[ooff:], dxb[off:]
    assert gn.fwd_ex_raw(x0, s, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y0, os_, mean, rstd,
                         ws) == gn.GN_OK
    assert gn.bwd_ex_raw(dy0, os_, x0, s, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx0, s,
                         dg, db, ws) == gn.GN_OK
    torch.cuda.synchronize()
    checks.assert_out("y", _dense(_view(yb, ooff, w, os_)), ref["y"], w.dtype)
    checks.assert_out("dx", _dense(_view(dxb, off, w, s)), ref["dx"], w.dtype)
    checks.assert_stat("mean", mean, ref["mean"])
    checks.assert_stat("rstd", rstd, ref["rstd"])
    checks.assert_param("dgamma", dg, ref["dgamma"])
    checks.assert_param("dbeta", db, ref["dbeta"])
    assert _untouched(yb, w, ooff, os_) and _untouched(dxb, w, off, s)


@pytest.mark.parametrize("name,w", CASES[:2], ids=[c[0] for c in CASES[:2]])
def test_strided_in_place(name, w):
    """y over x and dx over dy, in the same strided views."""
    inp = synth.make_inputs(w, "cpu", seed=52)
    ref = _oracle(inp, w)
    dt = synth.DTYPES[w.dtype]
    tot, off, s = _geometry(w, "channel_slice")
    xb = _place(inp["x"].cuda(), w, tot, off, s, dt)
    keep = xb.clone()
    dyb = _place(inp["dy"].cuda(), w, tot, off, s, dt)
    gm, bt = inp["gamma"].cuda(), inp["beta"].cuda()
    mean = torch.empty(w.N * w.G, device="cuda")
    rstd = torch.empty(w.N * w.G, device="cuda")
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, dt)
    assert gn.fwd_ex_raw(xb[off:], s, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, xb[off:], s,
                         mean, rstd, ws) == gn.GN_OK
    torch.cuda.synchronize()
    checks.assert_out("y (in place)", _dense(_view(xb, off, w, s)), ref["y"], w.dtype)
    assert _untouched(xb, w, off, s)
    dg, db = torch.empty(w.C, device="cuda"), torch.empty(w.C, device="cuda")
    assert gn.bwd_ex_raw(dyb[off:], s, keep[off:], s, mean, rstd, gm, w.N, w.C, w.HW, w.G,
                         w.layout, dyb[off:], s, dg, db, ws) == gn.GN_OK
    torch.cuda.synchronize()
    checks.assert_out("dx (in place)", _dense(_view(dyb, off, w, s)), ref["dx"], w.dtype)
    checks.assert_param("dgamma", dg, ref["dgamma"])


def test_dense_strides_match_gn_fwd_bit_for_bit():
    w = synth.WORKLOADS[4].scaled(name="svd", N=4, H=12, W=12)
    inp = synth.make_inputs(w, "cuda", seed=53)
    x, gm, bt = inp["x"], inp["gamma"], inp["beta"]
    gn.set_regime(gn.REGIME_TWO_KERNEL)
    try:
        y1, m1, r1 = gn.forward(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps)
        y2 = torch.empty_like(x)
        m2 = torch.empty_like(m1)
        r2 = torch.empty_like(r1)
        ws = gn.alloc_workspace(gn.OP_FWD, w.N, w.C, w.HW, w.G, w.layout, x.dtype)
        s = (w.HW * w.C, w.C)
        assert gn.fwd_ex_raw(x, s, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y2, s, m2, r2,
                             ws) == gn.GN_OK
        torch.cuda.synchronize()
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    assert torch.equal(y1, y2) and torch.equal(m1, m2) and torch.equal(r1, r2)

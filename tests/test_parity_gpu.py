"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases (the oracle runs in well under a second) are compared element by
element; they span several CTAs, ragged row/chunk tails, both layouts, all
three dtypes, the 16-byte vector path and the scalar path.  The full-size
workloads are compared on sampled outputs plus the complete dgamma/dbeta.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from backward_normalization_gb300 import gn, synth
from tests import checks
from tests.cases import SPANNING, SPANNING_NAMES, strong_dy

pytestmark = pytest.mark.gpu

W = synth.BY_NAME


def _small_cases():
    c0, c1, c2, c3, c4 = synth.WORKLOADS
    return [
        ("fp32_nchw_2x32x16x16_g8", c0),
        ("fp16_nhwc_1x128x61x97_g16", c1.scaled(name="s1", H=61, W=97)),
        ("bf16_nhwc_3x320x17x17_g32", c2.scaled(name="s2", N=3, H=17, W=17)),
        ("fp32_nchw_3x64x48x48_g8", c3.scaled(name="s3", N=3, H=48, W=48)),
        ("fp32_nchw_2x64x47x49_g8_scalar", c3.scaled(name="s3b", N=2, H=47, W=49)),
        ("bf16_nhwc_4x512x12x12_g32_offsets", c4.scaled(name="s4", N=4, H=12, W=12)),
        ("fp16_nchw_2x24x20x20_g1_layernorm", c1.scaled(name="ln", layout="nchw", N=2, C=24, G=1, H=20, W=20)),
        ("bf16_nhwc_2x48x5x10_g48_instancenorm", c2.scaled(name="in", N=2, C=48, G=48, H=5, W=10)),
        ("fp16_nhwc_3x6x7x11_g3_scalar", c1.scaled(name="sc", N=3, C=6, G=3, H=7, W=11)),
        ("fp32_nchw_5x12x1x1_g4", c0.scaled(name="hw1", N=5, C=12, G=4, H=1, W=1)),
        ("bf16_nhwc_7x16x1x1_g4", c2.scaled(name="hw1b", N=7, C=16, G=4, H=1, W=1)),
        ("fp32_nchw_1x1x1x3_g1", c0.scaled(name="tiny", N=1, C=1, G=1, H=1, W=3)),
        ("fp16_nhwc_2x4096x5x8_g32_wide", c1.scaled(name="wide", N=2, C=4096, G=32, H=5, W=8)),
        ("fp32_nhwc_2x64x15x20_g8", c0.scaled(name="f32nhwc", layout="nhwc", C=64, H=15, W=20)),
        ("fp16_nchw_2x16x64x64_g4", c1.scaled(name="f16nchw", layout="nchw", N=2, C=16, G=4, H=64, W=64)),
        ("bf16_nchw_2x8x3x683_g2_scalar", c2.scaled(name="b16nchw", layout="nchw", N=2, C=8, G=2, H=3, W=683)),
        ("bf16_nhwc_1x32x300x300_g8_many_rows", c2.scaled(name="rows", N=1, C=32, G=8, H=300, W=300)),
        # many reduction units: pass-2 tasks of the pipelined kernel trail pass 1 by fewer units
        # than there are, so both passes of different units interleave in its task order
        ("fp32_nchw_16x64x48x48_g8_many_units", c3.scaled(name="mu3", N=16, H=48, W=48)),
        ("bf16_nhwc_40x64x48x48_g8_many_units", c4.scaled(name="mu4", N=40, C=64, G=8, H=48, W=48)),
        # groups of 80 channels across the two 600-channel column blocks: both blocks'
        # second-kernel CTAs derive the shared group's statistics
        ("fp32_nhwc_2x1200x2x3_g15_straddle", c0.scaled(name="strad", layout="nhwc", N=2, C=1200, G=15, H=2, W=3)),
        # blocks of 8 planes cut groups of 12 planes
        ("fp32_nchw_2x36x10x10_g3_row_blocks", c0.scaled(name="blk", N=2, C=36, G=3, H=10, W=10)),
        # fp64 storage (computed in fp32): row blocks, plane chunks, channels-last vectors
        # of two doubles that span groups (Cg = 5), and both scalar paths
        ("fp64_nchw_2x32x16x16_g8", c0.scaled(name="d0", dtype="f64")),
        ("fp64_nchw_2x16x64x64_g4", c0.scaled(name="d1", dtype="f64", C=16, G=4, H=64, W=64)),
        ("fp64_nhwc_3x40x9x11_g8", c0.scaled(name="d2", dtype="f64", layout="nhwc", N=3, C=40, G=8, H=9, W=11)),
        ("fp64_nchw_2x6x7x9_g3_scalar", c0.scaled(name="d3", dtype="f64", C=6, G=3, H=7, W=9)),
        ("fp64_nhwc_2x3x5x5_g3_scalar", c0.scaled(name="d4", dtype="f64", layout="nhwc", C=3, G=3, H=5, W=5)),
    ] + SPANNING


SMALL = _small_cases()
SMALL_BASE = [c for c in SMALL if c[1].name not in SPANNING_NAMES]

# Slices larger than shared memory: the resident regime streams part of each
# slice through its ring and reads it again in the second pass.
STREAMING = [
    ("fp32_nchw_1x16x512x512_g2_stream", synth.WORKLOADS[3].scaled(name="st3", N=1, C=16, G=2)),
    ("bf16_nhwc_2x320x64x64_g32_stream_bwd", synth.WORKLOADS[2].scaled(name="st2", N=2)),
    ("fp16_nchw_2x8x300x300_g1_stream", synth.WORKLOADS[1].scaled(name="st1", layout="nchw", N=2, C=8, G=1, H=300, W=300)),
]


REGIMES = {"auto": gn.REGIME_AUTO, "two_kernel": gn.REGIME_TWO_KERNEL, "resident": gn.REGIME_RESIDENT,
           "pipelined": gn.REGIME_PIPELINED, "wave": gn.REGIME_WAVE, "flat": gn.REGIME_FLAT}


@pytest.fixture(params=list(REGIMES))
def regime(request):
    """Runs a test under the automatic kernel choice and with each family
    forced, so both families see every case they can run."""
    gn.set_regime(REGIMES[request.param])
    yield request.param
    gn.set_regime(gn.REGIME_AUTO)


def _oracle_full(inp, w):
    o = oracle.get()
    L = synth.LAYOUTS[w.layout]
    x = inp["x"].double().numpy()
    dy = inp["dy"].double().numpy()
    g = inp["gamma"].double().numpy()
    b = inp["beta"].double().numpy()
    y, mean, rstd = o.forward(x, w.N, w.C, w.HW, w.G, L, g, b, w.eps)
    dx, dg, db = o.backward(dy, x, w.N, w.C, w.HW, w.G, L, g, w.eps)
    return dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)


def _gpu_run(inp, w, dev="cuda", gamma=True, beta=True, params=True):
    x = inp["x"].to(dev)
    dy = inp["dy"].to(dev)
    gm = inp["gamma"].to(dev) if gamma else None
    bt = inp["beta"].to(dev) if beta else None
    y, mean, rstd = gn.forward(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps)
    dx, dg, db = gn.backward(dy, x, mean, rstd, w.N, w.C, w.HW, w.G, w.layout, gm,
                             need_params=params)
    torch.cuda.synchronize()
    return dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)


def _compare(got, ref, w):
    checks.assert_out("y", got["y"], ref["y"], w.dtype)
    checks.assert_out("dx", got["dx"], ref["dx"], w.dtype)
    checks.assert_stat("mean", got["mean"], ref["mean"])
    checks.assert_stat("rstd", got["rstd"], ref["rstd"])
    if got["dgamma"] is not None:
        checks.assert_param("dgamma", got["dgamma"], ref["dgamma"])
        checks.assert_param("dbeta", got["dbeta"], ref["dbeta"])


@pytest.mark.parametrize("name,w", SMALL + STREAMING, ids=[c[0] for c in SMALL + STREAMING])
def test_small_parity(name, w, regime):
    inp = synth.make_inputs(w, "cpu", seed=0)
    if w.name in SPANNING_NAMES:
        inp = strong_dy(inp, w)
    got = _gpu_run(inp, w)
    _compare(got, _oracle_full(inp, w), w)


@pytest.mark.parametrize("name,w", SMALL[:6] + STREAMING[:2], ids=[c[0] for c in SMALL[:6] + STREAMING[:2]])
def test_bit_identical_runs(name, w, regime):
    inp = synth.make_inputs(w, "cpu", seed=1)
    a = _gpu_run(inp, w)
    b = _gpu_run(inp, w)
    for k in a:
        assert torch.equal(a[k].view(torch.uint8) if a[k].dtype != torch.float32 else a[k],
                           b[k].view(torch.uint8) if b[k].dtype != torch.float32 else b[k]), k


@pytest.mark.parametrize("name,w", [SMALL[1], SMALL[3], SMALL[0]], ids=["nhwc", "nchw_m0", "nchw_m1"])
def test_no_affine_and_output_mask(name, w, regime):
    inp = synth.make_inputs(w, "cpu", seed=2)
    got = _gpu_run(inp, w, gamma=False, beta=False, params=False)
    o = oracle.get()
    L = synth.LAYOUTS[w.layout]
    x, dy = inp["x"].double().numpy(), inp["dy"].double().numpy()
    y, mean, rstd = o.forward(x, w.N, w.C, w.HW, w.G, L, None, None, w.eps)
    dx, dg, db = o.backward(dy, x, w.N, w.C, w.HW, w.G, L, None, w.eps)
    checks.assert_out("y", got["y"], y, w.dtype)
    checks.assert_out("dx", got["dx"], dx, w.dtype)
    checks.assert_stat("rstd", got["rstd"], rstd)
    # gamma given but beta absent: beta = 0
    inp2 = dict(inp)
    got2 = _gpu_run(inp2, w, gamma=True, beta=False)
    y2, _, _ = o.forward(x, w.N, w.C, w.HW, w.G, L, inp["gamma"].double().numpy(), None, w.eps)
    checks.assert_out("y(no beta)", got2["y"], y2, w.dtype)


@pytest.mark.parametrize("name,w", [SMALL[1], SMALL[2], SMALL[3], SMALL[0]],
                         ids=["nhwc", "nhwc_spanning", "nchw_m0", "nchw_m1"])
def test_single_parameter_gradient_masks(name, w, regime):
    """dgamma alone (dbeta NULL) and dbeta alone (dgamma NULL): the requested
    gradient and dx match the oracle."""
    inp = synth.make_inputs(w, "cpu", seed=8)
    ref = _oracle_full(inp, w)
    dev = "cuda"
    x, dy = inp["x"].to(dev), inp["dy"].to(dev)
    gm, bt = inp["gamma"].to(dev), inp["beta"].to(dev)
    y, mean, rstd = gn.forward(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps)
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, x.dtype)
    for want_g in (True, False):
        dx = torch.empty_like(x)
        out = torch.full((w.C,), 5.0, device=dev)
        dg, db = (out, None) if want_g else (None, out)
        rc = gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws)
        assert rc == gn.GN_OK
        torch.cuda.synchronize()
        checks.assert_out("dx", dx, ref["dx"], w.dtype)
        checks.assert_param("dgamma" if want_g else "dbeta", out,
                            ref["dgamma"] if want_g else ref["dbeta"])


@pytest.mark.parametrize("name,w", [SMALL[1], SMALL[3]], ids=["nhwc", "nchw"])
def test_misaligned_pointers_take_scalar_path(name, w):
    """Buffers offset by one element (not 16-byte aligned) still give the
    right answer (the scalar path)."""
    inp = synth.make_inputs(w, "cpu", seed=3)
    dev = "cuda"
    E = w.E
    dt = synth.DTYPES[w.dtype]
    xb = torch.empty(E + 1, dtype=dt, device=dev)
    dyb = torch.empty(E + 1, dtype=dt, device=dev)
    yb = torch.empty(E + 1, dtype=dt, device=dev)
    dxb = torch.empty(E + 1, dtype=dt, device=dev)
    x, dy, y, dx = xb[1:], dyb[1:], yb[1:], dxb[1:]
    x.copy_(inp["x"])
    dy.copy_(inp["dy"])
    gm, bt = inp["gamma"].to(dev), inp["beta"].to(dev)
    mean = torch.empty(w.N * w.G, device=dev)
    rstd = torch.empty(w.N * w.G, device=dev)
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, dt)
    assert gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd, ws) == 0
    dg = torch.empty(w.C, device=dev)
    db = torch.empty(w.C, device=dev)
    assert gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws) == 0
    torch.cuda.synchronize()
    assert gn.plan_info(0, w.N, w.C, w.HW, w.G, w.layout, dt, aligned=False).vector_width == 1
    _compare(dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db), _oracle_full(inp, w), w)


@pytest.mark.parametrize("name,w", [SMALL[2], SMALL[3]], ids=["nhwc", "nchw"])
def test_in_place(name, w, regime):
    """y may overwrite x, and dx may overwrite dy."""
    inp = synth.make_inputs(w, "cpu", seed=4)
    ref = _oracle_full(inp, w)
    dev = "cuda"
    x = inp["x"].to(dev)
    gm, bt = inp["gamma"].to(dev), inp["beta"].to(dev)
    mean = torch.empty(w.N * w.G, device=dev)
    rstd = torch.empty(w.N * w.G, device=dev)
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, x.dtype)
    x_keep = x.clone()
    assert gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, x, mean, rstd, ws) == 0
    torch.cuda.synchronize()
    checks.assert_out("y(in place)", x, ref["y"], w.dtype)
    dy = inp["dy"].to(dev)
    dg = torch.empty(w.C, device=dev)
    db = torch.empty(w.C, device=dev)
    assert gn.bwd_raw(dy, x_keep, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dy, dg, db, ws) == 0
    torch.cuda.synchronize()
    checks.assert_out("dx(in place)", dy, ref["dx"], w.dtype)
    checks.assert_param("dgamma", dg, ref["dgamma"])


def test_workspace_reuse_and_canaries(regime):
    """The workspace's contents are dead between calls: refilled with random
    bytes before every call, it gives the same bits as the first call; the
    error word reads clear; nothing is written past the end of the workspace
    or of any output."""
    w = SMALL[5][1]
    inp = synth.make_inputs(w, "cpu", seed=5)
    ref = _oracle_full(inp, w)
    dev = "cuda"
    dt = synth.DTYPES[w.dtype]
    pad = 64
    n_ws = gn.workspace_size(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, dt)
    n_ws = max(n_ws, gn.workspace_size(gn.OP_FWD, w.N, w.C, w.HW, w.G, w.layout, dt))
    wsb = torch.randint(0, 256, (n_ws + 256,), dtype=torch.uint8, device=dev)
    canary_ws = wsb[n_ws:].clone()
    ws = wsb[:n_ws]
    gen = torch.Generator(device=dev).manual_seed(55)

    def padded(n, dtype):
        b = torch.full((n + 2 * pad,), 7.0, dtype=dtype, device=dev)
        return b, b[pad:pad + n]

    yb, y = padded(w.E, dt)
    dxb, dx = padded(w.E, dt)
    mb, mean = padded(w.N * w.G, torch.float32)
    rb, rstd = padded(w.N * w.G, torch.float32)
    gb, dg = padded(w.C, torch.float32)
    bb, db = padded(w.C, torch.float32)
    x, dy = inp["x"].to(dev), inp["dy"].to(dev)
    gm, bt = inp["gamma"].to(dev), inp["beta"].to(dev)
    first = None
    for _ in range(3):
        ws.copy_(torch.randint(0, 256, (n_ws,), dtype=torch.uint8, device=dev, generator=gen))
        assert gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd, ws) == 0
        ws.copy_(torch.randint(0, 256, (n_ws,), dtype=torch.uint8, device=dev, generator=gen))
        assert gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws) == 0
        assert gn.workspace_status(ws) == gn.GN_OK
        got = [t.clone() for t in (y, mean, rstd, dx, dg, db)]
        if first is None:
            first = got
        for a, b in zip(first, got):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    assert torch.equal(wsb[n_ws:], canary_ws)
    for b in (yb, dxb, mb, rb, gb, bb):
        assert torch.all(b[:pad] == 7.0) and torch.all(b[-pad:] == 7.0)
    _compare(dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db), ref, w)


def test_workspace_shared_by_fwd_and_bwd(regime):
    """A forward and its backward (twice over) on one workspace give the same
    bits as calls on fresh workspaces.  At this shape the backward's plan uses
    more counters than the forward's (level-1 merges of its shorter chunks), so
    a layout that followed each op's own plan would put the backward's counters
    on the forward's partial records."""
    w = synth.WORKLOADS[3].scaled(name="fb3", N=2)
    dev = "cuda"
    inp = synth.make_inputs(w, dev, seed=7)
    x, dy, gm, bt = inp["x"], inp["dy"], inp["gamma"], inp["beta"]
    ref = _gpu_run(inp, w)
    dt = x.dtype
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, dt)
    for _ in range(2):
        y, mean, rstd = gn.forward(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, workspace=ws)
        dx, dg, db = gn.backward(dy, x, mean, rstd, w.N, w.C, w.HW, w.G, w.layout, gm, workspace=ws)
        torch.cuda.synchronize()
        got = dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)
        for k in got:
            assert torch.equal(got[k], ref[k]), k
    assert gn.workspace_status(ws) == gn.GN_OK


def test_shared_workspace_across_shapes(regime):
    """One buffer, filled with random bytes once and never cleared, serves
    calls of different shapes in a row (each call clears its own counters)."""
    dev = "cuda"
    cases = [SMALL[0][1], SMALL[2][1], SMALL[3][1], SMALL[2][1], SMALL[5][1], SMALL[0][1]]
    n_ws = max(gn.workspace_size(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
               for w in cases for op in (0, 1))
    ws = torch.randint(0, 256, (n_ws,), dtype=torch.uint8, device=dev)
    for i, w in enumerate(cases):
        inp = synth.make_inputs(w, "cpu", seed=10 + i)
        x, dy = inp["x"].to(dev), inp["dy"].to(dev)
        gm, bt = inp["gamma"].to(dev), inp["beta"].to(dev)
        y, mean, rstd = gn.forward(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, workspace=ws)
        dx, dg, db = gn.backward(dy, x, mean, rstd, w.N, w.C, w.HW, w.G, w.layout, gm, workspace=ws)
        torch.cuda.synchronize()
        _compare(dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db), _oracle_full(inp, w), w)


FINALISATION = [
    # (case, finalised in the second kernel, items per level-1 record)
    ("fp16_nhwc_1x128x64x64_g16_chain_level1", synth.WORKLOADS[1].scaled(name="f2l1", H=64, W=64), 0, 8),
    ("fp16_nhwc_1x2048x32x32_g32_chain", synth.WORKLOADS[1].scaled(name="f2ch", C=2048, G=32, H=32, W=32), 0, 8),
    ("bf16_nhwc_16x512x8x8_g32_chain", synth.WORKLOADS[4].scaled(name="f2c4", N=16, H=8, W=8), 0, 1),
    ("fp32_nchw_2x16x64x64_g4_records", synth.WORKLOADS[3].scaled(name="f2r", N=2, C=16, G=4, H=64, W=64), 1, 1),
    ("fp32_nchw_2x36x10x10_g3_row_blocks", synth.WORKLOADS[0].scaled(name="f2b", N=2, C=36, G=3, H=10, W=10), 1, 1),
]


@pytest.mark.parametrize("name,w,fin2,l1", FINALISATION, ids=[c[0] for c in FINALISATION])
def test_finalisation_paths(name, w, fin2, l1):
    """Both places of the finalisation (the second kernel's CTAs from the
    records, or the first kernel's last arrival) and both record levels, on
    the two-kernel path, element by element against the oracle; repeated
    calls are bit-identical."""
    gn.set_regime(gn.REGIME_TWO_KERNEL)
    try:
        for op in (gn.OP_FWD, gn.OP_BWD):
            d = gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
            assert (d.regime, d.finalise_second, d.level1_items) == (0, fin2, l1)
        inp = synth.make_inputs(w, "cpu", seed=5)
        a = _gpu_run(inp, w)
        b = _gpu_run(inp, w)
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    _compare(a, _oracle_full(inp, w), w)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_zero_extents():
    dev = "cuda"
    x = torch.empty(0, device=dev)
    mean = torch.empty(0, device=dev)
    assert gn.fwd_raw(x, 0, 8, 16, 2, "nchw", None, None, 1e-5, x, mean, mean, None) == 0
    dg = torch.full((8,), 3.0, device=dev)
    db = torch.full((8,), 3.0, device=dev)
    assert gn.bwd_raw(x, x, mean, mean, None, 4, 8, 0, 2, "nhwc", x, dg, db, None) == 0
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(db == 0)


def test_constant_group_gives_beta(regime):
    """A constant group: xhat = 0, so y = beta and rstd = 1/sqrt(eps)."""
    w = SMALL[0][1]
    inp = synth.make_inputs(w, "cpu", seed=6)
    inp["x"] = torch.full_like(inp["x"], 1.5)
    got = _gpu_run(inp, w)
    ref = _oracle_full(inp, w)
    checks.assert_out("y", got["y"], ref["y"], w.dtype)
    checks.assert_stat("rstd", got["rstd"], ref["rstd"])
    checks.assert_out("dx", got["dx"], ref["dx"], w.dtype)


# ------------------------------------------------------------- full sizes
# The two small channels-last workloads are compared element by element in
# full; the two large ones at sampled offsets chosen per (n, g) group and at
# the boundaries of the plan's items or pieces (see _boundary_offsets).
# Mid-size NCHW problems that the automatic choice gives to the wave regime,
# with units of 2 MiB, 256 KiB, 128 KiB and 8 MiB, and pieces per unit (32,
# 56) that do not divide the CTA count, so units straddle two steps.
# Compared in full.
_AFFINE = dict(gamma=("normal", 1.0, 0.1), beta=("normal", 0.0, 0.1))
MID_WAVE = [
    ("fp32_nchw_4x64x256x256_g8", synth.WORKLOADS[3].scaled(name="mw0", N=4, H=256, W=256, **_AFFINE)),
    ("bf16_nchw_16x64x128x128_g8", synth.WORKLOADS[3].scaled(name="mw1", dtype="bf16", N=16, H=128, W=128,
                                                             **_AFFINE)),
    ("fp16_nchw_8x32x256x256_g32", synth.WORKLOADS[3].scaled(name="mw2", dtype="f16", N=8, C=32, G=32,
                                                             H=256, W=256, **_AFFINE)),
    # 8 MiB units over every CTA: 8 pieces per CTA cycle through the hold buffers
    ("fp32_nchw_2x32x512x512_g4", synth.WORKLOADS[3].scaled(name="mw3", N=2, C=32, G=4, **_AFFINE)),
]


@pytest.mark.parametrize("name,w", MID_WAVE, ids=[c[0] for c in MID_WAVE])
def test_mid_size_wave(name, w):
    plans = [gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype) for op in (0, 1)]
    assert all(d.regime == gn.REGIME_WAVE and d.hold_buffers >= 2 for d in plans)
    inp = synth.make_inputs(w, "cpu", seed=3)
    got = _gpu_run(inp, w)
    _compare(got, _oracle_full(inp, w), w)


def test_mid_size_wave_straddles():
    w = MID_WAVE[0][1]
    d = [gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype) for op in (0, 1)]
    assert any(x.ctas % x.pieces_per_unit != 0 for x in d)


# Channels-last problems on the flat regime, compared in full: runs that cut
# samples at odd rows (fp16, 1536 rows per sample), fp32 vectors of four
# channels with two samples in many runs, and one whose runs (441 KiB) exceed
# shared memory, so that both passes stream through the ring and pass 2 reads
# most chunks again.
MID_FLAT = [
    ("fp16_nhwc_8x320x32x48_g32", synth.WORKLOADS[2].scaled(name="mf0", dtype="f16", H=32, W=48)),
    ("fp32_nhwc_16x256x24x24_g16", synth.WORKLOADS[4].scaled(name="mf1", dtype="f32", N=16, C=256, G=16,
                                                             H=24, W=24)),
    ("bf16_nhwc_4x512x128x128_g32_ring", synth.WORKLOADS[4].scaled(name="mf2", N=4, H=128, W=128)),
    ("bf16_nhwc_300x64x1x2_g8_many_samples", synth.WORKLOADS[4].scaled(name="mf3", N=300, C=64, G=8,
                                                                       H=1, W=2)),
]


@pytest.mark.parametrize("name,w", MID_FLAT, ids=[c[0] for c in MID_FLAT])
def test_mid_size_flat(name, w):
    gn.set_regime(gn.REGIME_FLAT)
    try:
        plans = [gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype) for op in (0, 1)]
        assert all(d.regime == gn.REGIME_FLAT for d in plans)
        inp = synth.make_inputs(w, "cpu", seed=4)
        got = _gpu_run(inp, w)
        again = _gpu_run(inp, w)
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    _compare(got, _oracle_full(inp, w), w)
    for k in got:
        assert torch.equal(got[k], again[k]), k


FULL_COMPARE = {"bf16_nhwc_8x320x64x64_g32", "bf16_nhwc_32x512x32x32_g32"}


def _boundary_offsets(w, plans, per_group=8, seed=0, max_planes=64):
    """Flat offsets to check at full size:
      * per (n, g) group: its first and last element and per_group random ones;
      * NCHW: the first and last element of every channel plane, and, in
        max_planes planes (the first, the last and random ones), both sides
        of every item / piece boundary of each plan;
      * NHWC: at both rows around every item / piece boundary of each plan,
        in every sample, the first and last channel of every group."""
    rng = np.random.default_rng(seed)
    N, C, HW, G = w.N, w.C, w.HW, w.G
    Cg = C // G
    out = []
    n = np.repeat(np.arange(N), G)
    g = np.tile(np.arange(G), N)
    if w.layout == "nchw":
        lo = (n * C + g * Cg) * HW
        span = Cg * HW
        out += [lo, lo + span - 1]
        out += [lo + rng.integers(0, span, lo.size) for _ in range(per_group)]
        planes = np.arange(N * C) * HW
        out += [planes, planes + HW - 1]
        pick = np.unique(np.concatenate([[0, N * C - 1], rng.integers(0, N * C, max_planes)]))
        for d in plans:
            L = int(d.piece_elems)
            if 0 < L < HW:
                cuts = np.arange(L, HW, L)
                for pl in pick:
                    out += [pl * HW + cuts - 1, pl * HW + cuts]
    else:
        first = n * HW * C + g * Cg
        last = (n * HW + HW - 1) * C + (g + 1) * Cg - 1
        out += [first, last]
        for _ in range(per_group):
            hw = rng.integers(0, HW, n.size)
            c = g * Cg + rng.integers(0, Cg, n.size)
            out.append((n * HW + hw) * C + c)
        chans = np.concatenate([np.arange(G) * Cg, np.arange(G) * Cg + Cg - 1])
        for d in plans:
            rb = int(d.piece_elems)
            if 0 < rb < HW:
                rows = np.concatenate([np.arange(rb, HW, rb) - 1, np.arange(rb, HW, rb)])
                for nn in range(N):
                    out.append(((nn * HW + rows[:, None]) * C + chans[None, :]).reshape(-1))
    idx = np.unique(np.concatenate([np.asarray(a, dtype=np.int64).reshape(-1) for a in out]))
    assert idx.min() >= 0 and idx.max() < w.E
    return idx


def _oracle_by_samples(w, inp, idx=None):
    """Oracle results for the whole batch, computed a block of samples at a
    time (sample n's statistics depend on sample n only): full y and dx when
    idx is None, else y and dx at the flat offsets idx; mean/rstd/dgamma/
    dbeta in full."""
    o = oracle.get()
    L = synth.LAYOUTS[w.layout]
    gm = inp["gamma"].double().cpu().numpy()
    bt = inp["beta"].double().cpu().numpy()
    per_n = w.C * w.HW
    chunk_n = max(1, min(w.N, (1 << 27) // per_n))  # at most ~128M elements per oracle call
    r = dict(mean=np.zeros(w.N * w.G), rstd=np.zeros(w.N * w.G), dgamma=np.zeros(w.C),
             dbeta=np.zeros(w.C))
    n_out = w.E if idx is None else idx.size
    r["y"] = np.zeros(n_out)
    r["dx"] = np.zeros(n_out)
    for n0 in range(0, w.N, chunk_n):
        n1 = min(w.N, n0 + chunk_n)
        lo, hi = n0 * per_n, n1 * per_n
        xs = inp["x"][lo:hi].double().cpu().numpy()
        dys = inp["dy"][lo:hi].double().cpu().numpy()
        if idx is None:
            ya, m, rs = o.forward(xs, n1 - n0, w.C, w.HW, w.G, L, gm, bt, w.eps)
            dxa, dg, db = o.backward(dys, xs, n1 - n0, w.C, w.HW, w.G, L, gm, w.eps)
            r["y"][lo:hi] = ya
            r["dx"][lo:hi] = dxa
        else:
            sel = (idx >= lo) & (idx < hi)
            ya, m, rs = o.forward_at(xs, n1 - n0, w.C, w.HW, w.G, L, gm, bt, w.eps, idx[sel] - lo)
            dxa, dg, db = o.backward_at(dys, xs, n1 - n0, w.C, w.HW, w.G, L, gm, w.eps,
                                        idx[sel] - lo)
            r["y"][sel] = ya
            r["dx"][sel] = dxa
        r["mean"][n0 * w.G:n1 * w.G] = m
        r["rstd"][n0 * w.G:n1 * w.G] = rs
        r["dgamma"] += dg
        r["dbeta"] += db
    return r


FULL = ([(w, "auto") for w in synth.WORKLOADS[1:]]
        + [(synth.WORKLOADS[3], "two_kernel"), (synth.WORKLOADS[2], "resident"),
           (synth.WORKLOADS[4], "two_kernel"), (synth.WORKLOADS[2], "two_kernel"),
           (synth.WORKLOADS[2], "flat"), (synth.WORKLOADS[4], "flat")])


@pytest.mark.parametrize("w,reg", FULL, ids=[f"{w.name}-{r}" for w, r in FULL])
def test_full_size(w, reg):
    """The benchmarked workloads at full size, in the launch configuration
    the benchmark times: y and dx in full (small workloads) or at per-group
    and plan-boundary offsets (large ones), with the relative L2 error of the
    whole of dx against the rounding bound on the small ones; mean, rstd,
    dgamma and dbeta in full; plus a bit-identical rerun."""
    dev = "cuda"
    gn.set_regime(REGIMES[reg])
    try:
        plans = [gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype) for op in (0, 1)]
        inp = synth.make_inputs(w, dev, seed=0)
        got = _gpu_run(inp, w)
        again = _gpu_run(inp, w)
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    for k in ("y", "dx"):
        assert torch.equal(got[k].view(torch.uint8) if got[k].dtype != torch.float32 else got[k],
                           again[k].view(torch.uint8) if again[k].dtype != torch.float32 else again[k]), k
    for k in ("mean", "rstd", "dgamma", "dbeta"):
        assert torch.equal(got[k], again[k]), k
    del again
    if w.name in FULL_COMPARE:
        ref = _oracle_by_samples(w, inp)
        checks.assert_out("y", got["y"], ref["y"], w.dtype)
        checks.assert_out("dx", got["dx"], ref["dx"], w.dtype)
        checks.assert_out_l2("y", got["y"], ref["y"], w.dtype)
        checks.assert_out_l2("dx", got["dx"], ref["dx"], w.dtype)
    else:
        idx = _boundary_offsets(w, plans)
        ref = _oracle_by_samples(w, inp, idx)
        it = torch.from_numpy(idx).to(dev)
        checks.assert_out("y", got["y"][it], ref["y"], w.dtype)
        checks.assert_out("dx", got["dx"][it], ref["dx"], w.dtype)
    checks.assert_stat("mean", got["mean"], ref["mean"])
    checks.assert_stat("rstd", got["rstd"], ref["rstd"])
    checks.assert_param("dgamma", got["dgamma"], ref["dgamma"])
    checks.assert_param("dbeta", got["dbeta"], ref["dbeta"])

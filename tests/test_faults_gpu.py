"""Failure detection on the GPU, without faulting it.

Two host-made failures: GN_FAULT_LAUNCH makes a call fail before it
enqueues anything; GN_FAULT_STALL makes one wave-regime call withhold one
piece's arrival (one flat-regime call, one chunk copy of CTA 0), so that the
waits on it run out (each wait is bounded, about 0.5 s) and the kernel
returns with the workspace's error word set.  In both cases the caller is told (the status, or gn_workspace_status),
the CUDA context stays usable, and the next call is correct.
"""
from __future__ import annotations

import time

import pytest
import torch

import oracle
from backward_normalization_gb300 import gn, synth
from tests import checks

pytestmark = pytest.mark.gpu

# wave-regime problems whose units are split over several CTAs: channels-last
# (stage B merges), and NCHW (the merge warp merges; several pieces per CTA,
# so stage A also waits for hold buffers)
W = synth.WORKLOADS[2].scaled(name="fault2", N=2, H=32, W=32)
W_NCHW = synth.WORKLOADS[3].scaled(name="fault3", N=2, H=256, W=256,
                                   gamma=("normal", 1.0, 0.1), beta=("normal", 0.0, 0.1))
# the flat regime: CTA 0 never gets its first chunk; the other CTAs read its
# (missing) records and finish
W_FLAT = synth.WORKLOADS[4].scaled(name="fault4", N=8, H=32, W=32)
CASES = [pytest.param(W, "wave", id="nhwc"), pytest.param(W_NCHW, "wave", id="nchw"),
         pytest.param(W_FLAT, "flat", id="flat_nhwc")]
REG = {"wave": gn.REGIME_WAVE, "flat": gn.REGIME_FLAT}


def _oracle(inp, w):
    o = oracle.get()
    L = synth.LAYOUTS[w.layout]
    x, dy = inp["x"].double().numpy(), inp["dy"].double().numpy()
    g, b = inp["gamma"].double().numpy(), inp["beta"].double().numpy()
    y, mean, rstd = o.forward(x, w.N, w.C, w.HW, w.G, L, g, b, w.eps)
    dx, dg, db = o.backward(dy, x, w.N, w.C, w.HW, w.G, L, g, w.eps)
    return dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)


@pytest.fixture
def forced():
    yield lambda reg: gn.set_regime(REG[reg])
    gn.set_regime(gn.REGIME_AUTO)
    gn.set_fault_injection(gn.FAULT_NONE)


def _calls(inp, w, ws):
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    gm, bt = inp["gamma"].cuda(), inp["beta"].cuda()
    y = torch.full_like(x, 3.0)
    mean = torch.empty(w.N * w.G, device="cuda")
    rstd = torch.empty(w.N * w.G, device="cuda")
    rc_f = gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd, ws)
    st_f = gn.workspace_status(ws)
    dx = torch.empty_like(x)
    dg, db = torch.empty(w.C, device="cuda"), torch.empty(w.C, device="cuda")
    rc_b = gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws)
    st_b = gn.workspace_status(ws)
    return (rc_f, st_f, rc_b, st_b), dict(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)


@pytest.mark.parametrize("w,reg", CASES)
def test_stalled_unit_is_reported_and_the_next_call_is_correct(forced, w, reg):
    forced(reg)
    for op in (gn.OP_FWD, gn.OP_BWD):
        d = gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
        assert d.regime == REG[reg] and d.pieces_per_unit > 1
    inp = synth.make_inputs(w, "cpu", seed=31)
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
    gn.set_fault_injection(gn.FAULT_STALL)  # applies to the next call only: the forward
    t0 = time.perf_counter()
    (rc_f, st_f, rc_b, st_b), _ = _calls(inp, w, ws)
    took = time.perf_counter() - t0
    assert rc_f == gn.GN_OK and st_f == gn.GN_ERR_TIMEOUT
    assert took < 30.0  # the waits are bounded (about 0.5 s)
    # the backward after it ran normally on the same workspace (its mean and
    # rstd are garbage, but its own waits all completed)
    assert rc_b == gn.GN_OK and st_b == gn.GN_OK
    # the next calls are correct, on the same workspace
    (rc_f, st_f, rc_b, st_b), got = _calls(inp, w, ws)
    assert (rc_f, st_f, rc_b, st_b) == (0, 0, 0, 0)
    ref = _oracle(inp, w)
    checks.assert_out("y", got["y"], ref["y"], w.dtype)
    checks.assert_out("dx", got["dx"], ref["dx"], w.dtype)
    checks.assert_stat("rstd", got["rstd"], ref["rstd"])
    checks.assert_param("dgamma", got["dgamma"], ref["dgamma"])


@pytest.mark.parametrize("w,reg", CASES)
def test_stalled_backward_is_reported(forced, w, reg):
    forced(reg)
    inp = synth.make_inputs(w, "cpu", seed=32)
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    gm, bt = inp["gamma"].cuda(), inp["beta"].cuda()
    y, mean, rstd = gn.forward(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, workspace=ws)
    assert gn.workspace_status(ws) == gn.GN_OK
    gn.set_fault_injection(gn.FAULT_STALL)
    dx = torch.empty_like(x)
    dg, db = torch.empty(w.C, device="cuda"), torch.empty(w.C, device="cuda")
    assert gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws) == 0
    assert gn.workspace_status(ws) == gn.GN_ERR_TIMEOUT
    assert gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws) == 0
    assert gn.workspace_status(ws) == gn.GN_OK
    ref = _oracle(inp, w)
    checks.assert_out("dx", dx, ref["dx"], w.dtype)
    checks.assert_param("dbeta", db, ref["dbeta"])


def test_launch_fault_enqueues_nothing():
    w = synth.WORKLOADS[0]
    inp = synth.make_inputs(w, "cuda", seed=33)
    x, gm, bt = inp["x"], inp["gamma"], inp["beta"]
    y = torch.full_like(x, 3.0)
    mean = torch.full((w.N * w.G,), 3.0, device="cuda")
    rstd = torch.full((w.N * w.G,), 3.0, device="cuda")
    ws = gn.alloc_workspace(gn.OP_FWD, w.N, w.C, w.HW, w.G, w.layout, x.dtype)
    gn.set_fault_injection(gn.FAULT_LAUNCH)
    try:
        rc = gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd, ws)
    finally:
        gn.set_fault_injection(gn.FAULT_NONE)
    assert rc == gn.GN_ERR_CUDA
    torch.cuda.synchronize()
    assert torch.all(y == 3.0) and torch.all(mean == 3.0)
    assert gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd, ws) == 0
    torch.cuda.synchronize()
    assert not torch.all(y == 3.0)

"""The batch split over data-parallel ranks, emulated on one GPU.

Each "rank" runs gn_fwd and gn_bwd through the C ABI on its own block of
samples (a contiguous slice of the batch in both layouts); the per-rank
dgamma/dbeta are then added in rank order with the same function the
multi-process path uses.  y, mean, rstd and dx of every shard, and the summed
parameter gradients, must match the fp64 oracle on the whole batch within
the parity tolerances (bit-equality with the unsharded call is not expected:
the summation order of dgamma/dbeta differs).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from backward_normalization_gb300 import gn, replicas, synth
from tests import checks

pytestmark = pytest.mark.gpu

CASES = [
    ("bf16_nhwc_8x512x16x16_g32", synth.WORKLOADS[4].scaled(name="sh4", N=8, H=16, W=16), 4),
    ("fp32_nchw_6x64x64x64_g8", synth.WORKLOADS[3].scaled(name="sh3", N=6, H=64, W=64), 3),
    ("bf16_nhwc_4x320x32x32_g32", synth.WORKLOADS[2].scaled(name="sh2", N=4, H=32, W=32), 2),
]


@pytest.mark.parametrize("name,w,ranks", CASES, ids=[c[0] for c in CASES])
def test_sharded_batch_matches_whole_batch(name, w, ranks):
    inp = synth.make_inputs(w, "cpu", seed=41)
    dev = "cuda"
    x, dy = inp["x"].to(dev), inp["dy"].to(dev)
    gm, bt = inp["gamma"].to(dev), inp["beta"].to(dev)
    per = w.N // ranks
    assert per * ranks == w.N
    ws_n = w.scaled(N=per)
    y, dx = torch.empty_like(x), torch.empty_like(x)
    mean = torch.empty(w.N * w.G, device=dev)
    rstd = torch.empty(w.N * w.G, device=dev)
    parts = []
    span = per * w.C * w.HW
    for r in range(ranks):
        sl = slice(r * span, (r + 1) * span)
        ms = slice(r * per * w.G, (r + 1) * per * w.G)
        ws = gn.alloc_workspace(gn.OP_BWD, per, w.C, w.HW, w.G, w.layout, x.dtype)
        assert gn.fwd_raw(x[sl], per, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y[sl], mean[ms],
                          rstd[ms], ws) == gn.GN_OK
        dg = torch.empty(w.C, device=dev)
        db = torch.empty(w.C, device=dev)
        assert gn.bwd_raw(dy[sl], x[sl], mean[ms], rstd[ms], gm, per, w.C, w.HW, w.G, w.layout,
                          dx[sl], dg, db, ws) == gn.GN_OK
        parts.append(torch.cat([dg, db]))
    tot = replicas.rank_order_sum(parts)
    torch.cuda.synchronize()
    assert ws_n.N == per
    o = oracle.get()
    L = synth.LAYOUTS[w.layout]
    xd, dyd = inp["x"].double().numpy(), inp["dy"].double().numpy()
    g, b = inp["gamma"].double().numpy(), inp["beta"].double().numpy()
    y_r, m_r, r_r = o.forward(xd, w.N, w.C, w.HW, w.G, L, g, b, w.eps)
    dx_r, dg_r, db_r = o.backward(dyd, xd, w.N, w.C, w.HW, w.G, L, g, w.eps)
    checks.assert_out("y", y, y_r, w.dtype)
    checks.assert_out("dx", dx, dx_r, w.dtype)
    checks.assert_stat("mean", mean, m_r)
    checks.assert_stat("rstd", rstd, r_r)
    checks.assert_param("dgamma", tot[:w.C], dg_r)
    checks.assert_param("dbeta", tot[w.C:], db_r)
    # and against the unsharded call
    _, _, _ = gn.forward(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps)
    dx1, dg1, db1 = gn.backward(dy, x, mean, rstd, w.N, w.C, w.HW, w.G, w.layout, gm)
    torch.cuda.synchronize()
    checks.assert_param("dgamma vs unsharded", tot[:w.C], checks.as_np(dg1))
    assert np.isfinite(checks.as_np(dx1)).all()

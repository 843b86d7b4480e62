"""GPU: the library's calls capture into a CUDA graph (the launch-bound small
problems replay without per-call launch cost) and replay bit-identically to
the eager calls, for every kernel family (two-kernel with programmatic
dependent launch, resident clusters, the cooperative wave and flat kernels,
rows)."""
from __future__ import annotations

import pytest
import torch

from backward_normalization_gb300 import gn, synth

pytestmark = pytest.mark.gpu

CASES = [
    ("bf16_nhwc_8x320x16x16_g32_resident", synth.WORKLOADS[2].scaled(name="g2", H=16, W=16),
     gn.REGIME_RESIDENT),
    ("bf16_nhwc_8x512x8x8_g32_two_kernel", synth.WORKLOADS[4].scaled(name="g4", N=8, H=8, W=8),
     gn.REGIME_TWO_KERNEL),
    ("fp32_nchw_4x64x48x48_g8_records", synth.WORKLOADS[3].scaled(name="g3", N=4, H=48, W=48),
     gn.REGIME_TWO_KERNEL),
    # one cooperative launch per op, units split over CTAs
    ("bf16_nhwc_8x320x16x16_g32_wave", synth.WORKLOADS[2].scaled(name="g2w", H=16, W=16),
     gn.REGIME_WAVE),
    ("fp32_nchw_4x64x48x48_g8_wave", synth.WORKLOADS[3].scaled(name="g3w", N=4, H=48, W=48),
     gn.REGIME_WAVE),
    # one cooperative launch per op with two grid barriers
    ("bf16_nhwc_8x320x16x16_g32_flat", synth.WORKLOADS[2].scaled(name="g2f", H=16, W=16),
     gn.REGIME_FLAT),
]


@pytest.fixture
def forced():
    yield gn.set_regime
    gn.set_regime(gn.REGIME_AUTO)


@pytest.mark.parametrize("name,w,regime", CASES, ids=[c[0] for c in CASES])
def test_groupnorm_graph_replay(name, w, regime, forced):
    forced(regime)
    for op in (gn.OP_FWD, gn.OP_BWD):
        assert gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype).regime == regime
    inp = synth.make_inputs(w, "cuda", seed=7)
    x, dy, gm, bt = inp["x"], inp["dy"], inp["gamma"], inp["beta"]
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, x.dtype)
    y, dx = torch.empty_like(x), torch.empty_like(x)
    mean = torch.empty(w.N * w.G, device="cuda")
    rstd = torch.empty_like(mean)
    dg, db = torch.empty(w.C, device="cuda"), torch.empty(w.C, device="cuda")

    def step(stream):
        assert gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd, ws,
                          stream) == 0
        assert gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws,
                          stream) == 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # eager, and the plan caches filled before capture
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (y, mean, rstd, dx, dg, db)]
    for t in (y, mean, rstd, dx, dg, db):
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (y, mean, rstd, dx, dg, db)):
        assert torch.equal(a, b)


def test_layernorm_graph_replay():
    w = synth.RowWorkload("graph_ln", "ln", "f16", 512, 1024)
    inp = synth.make_row_inputs(w, "cuda", seed=7)
    x, dy, gm, bt = inp["x"], inp["dy"], inp["gamma"], inp["beta"]
    M, N = w.M, w.N
    y, dx = torch.empty_like(x), torch.empty_like(x)
    mean, rstd = torch.empty(M, device="cuda"), torch.empty(M, device="cuda")
    dg, db = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    ws = torch.empty(gn.ln_workspace_size(M, N, "f16"), dtype=torch.uint8, device="cuda")

    def step(stream):
        assert gn.ln_fwd_raw(x, M, N, gm, bt, w.eps, y, mean, rstd, stream) == 0
        assert gn.ln_bwd_raw(dy, x, mean, rstd, gm, M, N, dx, dg, db, ws, stream) == 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (y, mean, rstd, dx, dg, db)]
    for t in (y, mean, rstd, dx, dg, db):
        t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step(side)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (y, mean, rstd, dx, dg, db)):
        assert torch.equal(a, b)

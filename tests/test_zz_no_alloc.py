"""gn_fwd_static_ws: the forward pass for callers that cannot allocate.

Serving code under a fixed memory budget, plugins without an allocator from
their host framework, and code where cudaMalloc is not allowed cannot hand
gn_fwd a workspace.  gn_fwd_static_ws takes no workspace and uses a scratch
array the library holds on each device.  These tests call it through the C
ABI, twice in a row (the second call finds the array holding the first
call's leftovers), and compare every output with gn_fwd's on the same inputs
within the parity tolerances.  The file is named so that pytest collects it
last.
"""
from __future__ import annotations

import pytest
import torch

from backward_normalization_gb300 import gn, synth
from tests import checks

pytestmark = pytest.mark.gpu

CASES = [
    # one kernel (a cluster holds each unit in shared memory)
    ("bf16_nhwc_4x512x12x12_g32", synth.WORKLOADS[4].scaled(name="na4", N=4, H=12, W=12)),
    # two kernels with workspace partial sums and arrival counters
    ("fp16_nhwc_1x128x61x97_g16", synth.WORKLOADS[1].scaled(name="na1", H=61, W=97)),
    ("fp32_nchw_2x32x16x16_g8", synth.WORKLOADS[0]),
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_static_workspace_matches_gn_fwd(name, w):
    gn.set_regime(gn.REGIME_AUTO)
    dev = "cuda"
    inp = synth.make_inputs(w, "cpu", seed=21)
    x = inp["x"].to(dev)
    gm, bt = inp["gamma"].to(dev), inp["beta"].to(dev)
    y_ref, mean_ref, rstd_ref = gn.forward(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps)
    torch.cuda.synchronize()
    for call in range(2):
        y = torch.full_like(x, 3.0)
        mean = torch.full((w.N * w.G,), 3.0, device=dev)
        rstd = torch.full((w.N * w.G,), 3.0, device=dev)
        rc = gn.fwd_static_ws_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd)
        assert rc == gn.GN_OK, gn.status_string(rc)
        torch.cuda.synchronize()
        checks.assert_out(f"y (call {call})", y, checks.as_np(y_ref), w.dtype)
        checks.assert_stat(f"mean (call {call})", mean, checks.as_np(mean_ref))
        checks.assert_stat(f"rstd (call {call})", rstd, checks.as_np(rstd_ref))


def test_static_workspace_rejects_problems_larger_than_the_array():
    gn.set_regime(gn.REGIME_AUTO)
    limit = 4 << 20
    # grow the batch of a small-plane problem until its workspace exceeds the array
    N = 1024
    while gn.workspace_size(gn.OP_FWD, N, 4096, 7, 32, "nhwc", "f16") <= limit:
        N *= 2
    fake = 1 << 20  # never dereferenced: the call is rejected before any launch
    rc = gn.lib().gn_fwd_static_ws(fake, N, 4096, 7, 32, 1, 1, None, None, 1e-5, fake * 2,
                                   fake * 3, fake * 4, None)
    assert rc == gn.GN_ERR_WORKSPACE

"""gn_fwd_static_ws: the forward pass for callers that cannot allocate.

Serving code under a fixed memory budget, plugins without an allocator from
their host framework, and code where cudaMalloc is not allowed cannot hand
gn_fwd a workspace.  gn_fwd_static_ws takes no workspace and uses a scratch
array the library holds on each device.  These tests call it through the C
ABI, twice in a row (the second call finds the array holding the first
call's leftovers), and compare every output with the fp64 oracle at the
parity tolerances.  The file is named so that pytest collects it last.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from backward_normalization_gb300 import gn, synth
from tests import checks

pytestmark = pytest.mark.gpu

LIMIT = 4 << 20  # GN_STATIC_WS_BYTES

CASES = [
    # one kernel (a cluster holds each unit in shared memory)
    ("bf16_nhwc_4x512x12x12_g32", synth.WORKLOADS[4].scaled(name="na4", N=4, H=12, W=12)),
    # two kernels with workspace partial sums and arrival counters
    ("fp16_nhwc_1x128x61x97_g16", synth.WORKLOADS[1].scaled(name="na1", H=61, W=97)),
    ("fp32_nchw_2x32x16x16_g8", synth.WORKLOADS[0]),
]


def _oracle_fwd(inp, w):
    o = oracle.get()
    return o.forward(inp["x"].double().numpy(), w.N, w.C, w.HW, w.G, synth.LAYOUTS[w.layout],
                     inp["gamma"].double().numpy(), inp["beta"].double().numpy(), w.eps)


def _static_call(inp, w, dev="cuda"):
    x = inp["x"].to(dev)
    gm, bt = inp["gamma"].to(dev), inp["beta"].to(dev)
    y = torch.full_like(x, 3.0)
    mean = torch.full((w.N * w.G,), 3.0, device=dev)
    rstd = torch.full((w.N * w.G,), 3.0, device=dev)
    rc = gn.fwd_static_ws_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd)
    assert rc == gn.GN_OK, gn.status_string(rc)
    torch.cuda.synchronize()
    return y, mean, rstd


def _check(tag, got, ref, w):
    y, mean, rstd = got
    yr, mr, rr = ref
    checks.assert_out(f"y ({tag})", y, yr, w.dtype)
    checks.assert_stat(f"mean ({tag})", mean, mr)
    checks.assert_stat(f"rstd ({tag})", rstd, rr)


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_static_workspace_matches_oracle(name, w):
    gn.set_regime(gn.REGIME_AUTO)
    inp = synth.make_inputs(w, "cpu", seed=21)
    ref = _oracle_fwd(inp, w)
    for call in range(2):
        _check(f"call {call}", _static_call(inp, w), ref, w)


def test_static_workspace_near_its_limit_after_another_shape():
    """A problem whose workspace is just under the array's size, run right
    after a problem of another shape left its partial records where the big
    problem keeps its arrival counters: every output still matches the
    oracle, twice in a row."""
    gn.set_regime(gn.REGIME_AUTO)
    base = synth.WORKLOADS[4].scaled(name="big", C=512, G=32, H=8, W=8)
    N = 16
    while gn.workspace_size(gn.OP_FWD, 2 * N, base.C, base.HW, base.G, base.layout, base.dtype) <= LIMIT:
        N *= 2
    lo, hi = N, 2 * N  # fits at lo, not at hi
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if gn.workspace_size(gn.OP_FWD, mid, base.C, base.HW, base.G, base.layout, base.dtype) <= LIMIT:
            lo = mid
        else:
            hi = mid
    big = base.scaled(N=lo)
    need = gn.workspace_size(gn.OP_FWD, big.N, big.C, big.HW, big.G, big.layout, big.dtype)
    assert LIMIT - 64 * 1024 < need <= LIMIT
    clear = gn.plan_info(gn.OP_FWD, big.N, big.C, big.HW, big.G, big.layout, big.dtype).clear_bytes
    assert clear > 256  # its counters reach past where a small problem's records start
    small = synth.WORKLOADS[0]
    s_inp = synth.make_inputs(small, "cpu", seed=22)
    b_inp = synth.make_inputs(big, "cpu", seed=23)
    s_ref = _oracle_fwd(s_inp, small)
    b_ref = _oracle_fwd(b_inp, big)
    for call in range(2):
        _check(f"small, call {call}", _static_call(s_inp, small), s_ref, small)
        _check(f"near the limit, call {call}", _static_call(b_inp, big), b_ref, big)


def test_static_workspace_rejects_problems_larger_than_the_array():
    gn.set_regime(gn.REGIME_AUTO)
    # grow the batch of a small-plane problem until its workspace exceeds the array
    N = 1024
    while gn.workspace_size(gn.OP_FWD, N, 4096, 7, 32, "nhwc", "f16") <= LIMIT:
        N *= 2
    fake = 1 << 20  # never dereferenced: the call is rejected before any launch
    rc = gn.lib().gn_fwd_static_ws(fake, N, 4096, 7, 32, 1, 1, None, None, 1e-5, fake * 2,
                                   fake * 3, fake * 4, None)
    assert rc == gn.GN_ERR_WORKSPACE

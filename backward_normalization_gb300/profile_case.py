"""Runs one GroupNorm workload through the C ABI a few times, with no timing,
as the target of a profiler capture.

The measured workloads are large (up to 2 GiB of inputs); a multi-pass
profiler capture wants the same kernels on a smaller case that still exceeds
the L2 cache.  This driver takes a workload by name and optionally overrides
its batch and spatial size, keeping its dtype, layout, channel count, group
count and value distributions:

    python -m backward_normalization_gb300.profile_case \\
        --workload fp16_nhwc_1x128x1024x2048_g16 --H 512 --calls 2

Each call is one forward followed by one backward on the same stream, so the
kernels launch in the order fwd-first, fwd-second, bwd-first, bwd-second
(one kernel per op in the resident, pipelined and wave regimes); every
regime but the wave regime first launches the small workspace-clear kernel.
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import gn, synth


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=[w.name for w in synth.WORKLOADS])
    ap.add_argument("--row-workload", choices=[w.name for w in synth.ROW_WORKLOADS],
                    help="a LayerNorm / RMSNorm row workload instead (--M overrides its rows)")
    ap.add_argument("--M", type=int)
    ap.add_argument("--N", type=int)
    ap.add_argument("--H", type=int)
    ap.add_argument("--W", type=int)
    ap.add_argument("--calls", type=int, default=2)
    ap.add_argument("--regime", choices=["auto", "two_kernel", "resident", "pipelined", "wave", "flat"],
                    default="auto")
    a = ap.parse_args(argv)
    if a.row_workload:
        return run_rows(a)
    if not a.workload:
        ap.error("--workload or --row-workload is required")
    w = synth.BY_NAME[a.workload]
    over = {k: v for k, v in (("N", a.N), ("H", a.H), ("W", a.W)) if v is not None}
    if over:
        w = w.scaled(**over)
    gn.set_regime({"auto": gn.REGIME_AUTO, "two_kernel": gn.REGIME_TWO_KERNEL,
                   "resident": gn.REGIME_RESIDENT, "pipelined": gn.REGIME_PIPELINED,
                   "wave": gn.REGIME_WAVE, "flat": gn.REGIME_FLAT}[a.regime])
    inp = synth.make_inputs(w, "cuda", seed=0)
    x, dy, gm, bt = inp["x"], inp["dy"], inp["gamma"], inp["beta"]
    y, dx = torch.empty_like(x), torch.empty_like(x)
    mean = torch.empty(w.N * w.G, device="cuda")
    rstd = torch.empty(w.N * w.G, device="cuda")
    dg = torch.empty(w.C, device="cuda")
    db = torch.empty(w.C, device="cuda")
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, x.dtype)
    stream = torch.cuda.current_stream()
    for _ in range(a.calls):
        rc = gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd, ws, stream)
        if rc != gn.GN_OK:
            raise gn.GnError(rc, "gn_fwd")
        rc = gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws,
                        stream)
        if rc != gn.GN_OK:
            raise gn.GnError(rc, "gn_bwd")
    torch.cuda.synchronize()
    pf = gn.plan_info(gn.OP_FWD, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
    pb = gn.plan_info(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
    print(f"{w.name} N={w.N} H={w.H} W={w.W}: {a.calls} calls, fwd launches {pf.launches} "
          f"(ctas {pf.ctas}), bwd launches {pb.launches} (ctas {pb.ctas})")
    return 0


def run_rows(a) -> int:
    """One row workload's forward then backward, --calls times."""
    w = synth.ROW_BY_NAME[a.row_workload]
    if a.M:
        w = synth.RowWorkload(w.name, w.op, w.dtype, a.M, w.N, w.eps)
    inp = synth.make_row_inputs(w, "cuda", seed=0)
    x, dy, gm, bt = inp["x"], inp["dy"], inp["gamma"], inp["beta"]
    for _ in range(a.calls):
        if w.op == "ln":
            y, mean, rstd = gn.ln_forward(x, w.M, w.N, gm, bt, w.eps)
            gn.ln_backward(dy, x, mean, rstd, w.M, w.N, gm)
        else:
            y, rstd = gn.rms_forward(x, w.M, w.N, gm, w.eps)
            gn.rms_backward(dy, x, rstd, w.M, w.N, gm)
    torch.cuda.synchronize()
    print(f"{w.name} M={w.M} N={w.N}: {a.calls} calls")
    return 0


if __name__ == "__main__":
    sys.exit(main())

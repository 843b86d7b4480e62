"""GroupNorm forward + backward benchmark on GB300.

One step = gn_fwd + gn_bwd (stats, normalize/affine, backward group
reduction, dx, dgamma/dbeta) over the fp16 channels_last workload
N=1, C=128, G=16, H=1024, W=2048 with inputs resident in HBM.  The metric is
achieved HBM bandwidth over the minimal traffic of the two ops
(forward: read x + write y; backward: read x, dy + write dx).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own copy of
the workload (weak scaling) and the per-channel dgamma/dbeta are summed across
ranks, in rank order, inside each step.  `--impl reference` times the fp64
CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "fp16_nhwc_1x128x1024x2048_g16"
METRIC = "GroupNorm fwd+bwd achieved HBM GB/s (% of GB300 roofline), us/call per config"
UNIT = "GB/s"
L2_FLUSH_BYTES = 512 << 20


def esize(dtype: str) -> int:
    return {"f32": 4, "f64": 8}.get(dtype, 2)


def min_bytes(w):
    """Minimal traffic per op: forward reads x and writes y; backward reads x
    and dy and writes dx."""
    e = w.E * esize(w.dtype)
    return {"fwd": 2 * e, "bwd": 3 * e}


REGIME_NAMES = {0: "two-kernel", 1: "resident", 2: "pipelined", 3: "wave", 4: "flat"}


def kernel_bytes(w, fwd_regime=0, bwd_regime=0):
    """Algorithmic bytes of each kernel (what it must move at least).  The
    two-kernel path reads its input twice by construction; the resident,
    pipelined, wave and flat regimes run one kernel per op that moves the op's
    minimal traffic."""
    e = w.E * esize(w.dtype)
    kb = {}
    if fwd_regime == 0:
        kb.update({"fwd_stats": e, "fwd_apply": 2 * e})
    else:
        kb["fwd_" + REGIME_NAMES[fwd_regime]] = 2 * e
    if bwd_regime == 0:
        kb.update({"bwd_reduce": 2 * e, "bwd_dx": 3 * e})
    else:
        kb["bwd_" + REGIME_NAMES[bwd_regime]] = 3 * e
    return kb


def kernel_times(kb, ev):
    """Per-kernel ms from the six events of one step (fwd: 0-2, bwd: 3-5)."""
    t = {}
    for k in kb:
        if k == "fwd_stats":
            t[k] = ev[0].elapsed_time(ev[1])
        elif k == "fwd_apply":
            t[k] = ev[1].elapsed_time(ev[2])
        elif k == "bwd_reduce":
            t[k] = ev[3].elapsed_time(ev[4])
        elif k == "bwd_dx":
            t[k] = ev[4].elapsed_time(ev[5])
        elif k.startswith("fwd_"):
            t[k] = ev[0].elapsed_time(ev[2])
        else:
            t[k] = ev[3].elapsed_time(ev[5])
    return t


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def config_of(w, extra=None):
    c = {"workload": w.name, "N": w.N, "C": w.C, "G": w.G, "H": w.H, "W": w.W,
         "layout": w.layout, "io_dtype": w.dtype, "eps": w.eps}
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile

            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[3][1:5])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in busy),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(busy), "power_w_max": max(r[2] for r in rows)}


# --------------------------------------------------------------- oracle leg
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """A bounded sample of a workload for timing the fp64 CPU oracle: the first
    `ns` samples of the batch (or, for a one-sample workload, its first `h`
    image rows), cut into its (sample, group) units.  Each unit is handed to
    the oracle as a one-group problem of its own -- the oracle's arithmetic
    for a group depends on that group's values only, so this is the same
    computation it does on the whole tensor, and units can run on separate
    host threads (ctypes releases the GIL during each oracle call).  The
    channels_last units are gathered into contiguous [HW, Cg] arrays before
    the clock starts (a layout copy, not part of the method)."""

    def __init__(self, w, ns=None, h=None, seed=0):
        from backward_normalization_gb300 import synth

        self.w = w.scaled(N=ns) if ns else w.scaled(H=h)
        ws = self.w
        inp = synth.make_inputs(ws, "cpu", seed=seed)
        x = inp["x"].double().numpy()
        dy = inp["dy"].double().numpy()
        gm = inp["gamma"].double().numpy()
        bt = inp["beta"].double().numpy()
        Cg = ws.C // ws.G
        self.units = []
        for n in range(ws.N):
            for g in range(ws.G):
                c0 = g * Cg
                if ws.layout == "nchw":
                    lo = (n * ws.C + c0) * ws.HW
                    xu, du = x[lo:lo + Cg * ws.HW], dy[lo:lo + Cg * ws.HW]
                else:
                    xs = x.reshape(ws.N, ws.HW, ws.C)[n, :, c0:c0 + Cg]
                    ds = dy.reshape(ws.N, ws.HW, ws.C)[n, :, c0:c0 + Cg]
                    xu, du = xs.copy().reshape(-1), ds.copy().reshape(-1)
                self.units.append((xu, du, gm[c0:c0 + Cg].copy(), bt[c0:c0 + Cg].copy(), Cg))
        self.layout = synth.LAYOUTS[ws.layout]
        mb = min_bytes(ws)
        self.bytes = mb["fwd"] + mb["bwd"]
        part = f"samples 0..{ws.N - 1}" if ns else f"image rows 0..{ws.H - 1}"
        self.desc = (f"fp64 oracle fwd+bwd on {part} of {w.name} ({ws.E} elements, "
                     f"{ws.E / w.E:.4f} of the workload), {len(self.units)} (sample, group) units")

    def run(self, threads: int) -> float:
        """Seconds for fwd + bwd of every unit on `threads` host threads."""
        import concurrent.futures as cf

        import oracle

        o = oracle.get()
        ws, L = self.w, self.layout

        def one(u):
            xu, du, g, b, Cg = u
            o.forward(xu, 1, Cg, ws.HW, 1, L, g, b, ws.eps)
            o.backward(du, xu, 1, Cg, ws.HW, 1, L, g, ws.eps)

        t0 = time.perf_counter()
        if threads <= 1:
            for u in self.units:
                one(u)
        else:
            with cf.ThreadPoolExecutor(max_workers=threads) as ex:
                list(ex.map(one, self.units))
        return time.perf_counter() - t0


def oracle_sample_for(w, target_s: float, threads: int = 1):
    """An OracleSample of w whose run on `threads` threads takes about
    target_s seconds here (sized from a small calibration run on as many
    threads)."""
    if w.N > 1:
        ns = min(w.N, max(1, threads // max(1, w.G)))
        probe = OracleSample(w, ns=ns)
        per = probe.run(threads) / ns
        ns = int(max(1, min(w.N, round(target_s / max(per, 1e-6)))))
        return OracleSample(w, ns=ns)
    probe = OracleSample(w, h=4)
    per = probe.run(threads) / 4
    h = int(max(1, min(w.H, round(target_s / max(per, 1e-6)))))
    return OracleSample(w, h=h)


def cpu_baselines(workloads, target_s=2.0):
    """Per workload: the oracle on one thread and on all host cores, over the
    same bounded sample (GB/s over the sample's minimal traffic)."""
    nt = host_cores()
    out = {}
    for w in workloads:
        smp = oracle_sample_for(w, target_s, 1)
        t1 = smp.run(1)
        tn = smp.run(nt)
        out[w.name] = {"single_thread_gbs": round(smp.bytes / t1 / 1e9, 4),
                       "all_cores_gbs": round(smp.bytes / tn / 1e9, 4), "cores": nt,
                       "seconds_single": round(t1, 3), "seconds_all_cores": round(tn, 3),
                       "sample": smp.desc}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from backward_normalization_gb300 import synth

    w = synth.BY_NAME[WORKLOAD]
    nt = host_cores()
    # the whole run stays within about two minutes: each step a bounded
    # sample of the workload, on all host cores
    smp = oracle_sample_for(w, min(0.5, 60.0 / (args.steps + args.warmup)), nt)
    for _ in range(args.warmup):
        smp.run(nt)
    times = [smp.run(nt) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = smp.bytes / (ms * 1e-3) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, {"sample": smp.desc}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt, "kind": "oracle",
                             "sample": smp.desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def traffic_from_profiles(kernel_key):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if the
    kernel sources are unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("src_sha") != source_sha():
        return None
    k = d.get("kernels", {}).get(kernel_key)
    return None if k is None else k.get("dram_bytes_per_launch")


def source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "backward_normalization_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def variant_workloads(synth):
    """The special cases of the op on the large workloads' shapes, timed beside
    them: InstanceNorm (G = C) and GroupNorm without affine parameters (gamma
    and beta absent, so no dgamma / dbeta either)."""
    c3, c4 = synth.BY_NAME["fp32_nchw_112x64x512x512_g8"], synth.BY_NAME["bf16_nhwc_32x512x32x32_g32"]
    return [(c4.scaled(name="bf16_nhwc_32x512x32x32_g512_instancenorm", G=512), True),
            (c3.scaled(name="fp32_nchw_16x64x512x512_g64_instancenorm", N=16, G=64), True),
            (c4.scaled(name="bf16_nhwc_32x512x32x32_g32_no_affine"), False),
            (c3.scaled(name="fp32_nchw_16x64x512x512_g8_no_affine", N=16), False)]


def time_configs(gn, synth, torch, flush, names=None, reps=20, variants=False):
    """Per-workload fwd and bwd times (median of reps, L2 flushed before each
    call) for the large workloads (and, with `variants`, the special cases of
    variant_workloads).  All reps are queued before the first
    synchronisation, so the GPU never waits for the host between calls."""
    out = {}
    peak, _ = load_peaks()
    stream = torch.cuda.current_stream()
    todo = []
    for w in synth.WORKLOADS[1:]:
        if not names:
            todo.append((w, True))
        for nm in names or ():
            base, _, nn = nm.partition(":")  # "workload" or "workload:N" (batch override)
            if base == w.name:
                todo.append((w.scaled(N=int(nn)) if nn else w, True))
    if variants:
        todo += variant_workloads(synth)
    for w, affine in todo:
        inp = synth.make_inputs(w, "cuda", seed=0)
        x, dy, gm, bt = inp["x"], inp["dy"], inp["gamma"], inp["beta"]
        if not affine:
            gm = bt = None
        y = torch.empty_like(x)
        dx = torch.empty_like(x)
        mean = torch.empty(w.N * w.G, device="cuda")
        rstd = torch.empty(w.N * w.G, device="cuda")
        dg = torch.empty(w.C, device="cuda") if affine else None
        db = torch.empty(w.C, device="cuda") if affine else None
        ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, x.dtype)
        n_it = reps + 3
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_it)]
        evk = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_it)]
        # first the op times (no event between an op's kernels, which would hold
        # back the second kernel's early launch), then per-kernel times
        for split, table in ((False, evs), (True, evk)):
            for it in range(n_it):
                ev = table[it]
                flush()
                gn.set_timing_events(ev[0], ev[1] if split else None, ev[2])
                assert gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd,
                                  ws, stream) == 0
                flush()
                gn.set_timing_events(ev[3], ev[4] if split else None, ev[5])
                assert gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db,
                                  ws, stream) == 0
                gn.set_timing_events()
        torch.cuda.synchronize()
        pf = gn.plan_info(0, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
        pb = gn.plan_info(1, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
        kb = kernel_bytes(w, pf.regime, pb.regime)
        rec = {"fwd": [], "bwd": []}
        for ev, ek in zip(evs[3:], evk[3:]):
            rec["fwd"].append(ev[0].elapsed_time(ev[2]))
            rec["bwd"].append(ev[3].elapsed_time(ev[5]))
            for k, v in kernel_times(kb, ek).items():
                rec.setdefault(k, []).append(v)
        mb = min_bytes(w)
        med = {k: statistics.median(v) for k, v in rec.items()}
        fwd_gbs = mb["fwd"] / (med["fwd"] * 1e-3) / 1e9
        bwd_gbs = mb["bwd"] / (med["bwd"] * 1e-3) / 1e9
        key = w.name if w.name not in synth.BY_NAME or w.N == synth.BY_NAME[w.name].N \
            else f"{w.name}:N={w.N}"
        out[key] = {
            "regime": {"fwd": REGIME_NAMES[pf.regime], "bwd": REGIME_NAMES[pb.regime]},
            "fwd_us": round(med["fwd"] * 1e3, 2), "bwd_us": round(med["bwd"] * 1e3, 2),
            "fwd_gbs": round(fwd_gbs, 1), "bwd_gbs": round(bwd_gbs, 1),
            "fwd_frac": round(fwd_gbs / peak, 4), "bwd_frac": round(bwd_gbs / peak, 4),
            "fwd_frac_of_8tbs": round(fwd_gbs / 8000.0, 4), "bwd_frac_of_8tbs": round(bwd_gbs / 8000.0, 4),
            "kernels_us": {k: round(med[k] * 1e3, 2) for k in kb},
            "kernels_frac": {k: round(kb[k] / (med[k] * 1e-3) / 1e9 / peak, 4) for k in kb},
        }
        del x, dy, y, dx, inp, ws
        torch.cuda.empty_cache()
    return out


# Context, not targets: the backward times the ROCm normalization-backward
# page reports for these shapes on an AMD Instinct MI350X ("Layer Norm
# Backward Benchmark" table, Tiled+Two pass column, average µs).
ROW_MI350X_BWD_US = {
    "ln_f16_4096x1024": 13.12, "ln_bf16_4096x1024": 13.10, "ln_f32_4096x1024": 15.90,
    "ln_f16_1024x768": 11.05, "ln_f16_131072x64": 27.70, "ln_bf16_131072x4096": 513.38,
    "ln_f16_8192x768": 16.56, "rms_f16_4096x1024": 11.18, "rms_bf16_131072x4096": 476.03,
    "rms_f16_131072x64": 17.29,
}


def time_rows(gn, synth, torch, flush, reps=20):
    """LayerNorm / RMSNorm over rows on the benchmark table's shapes: median
    fwd and bwd µs (L2 flushed before each call, events on the stream),
    GB/s over minimal traffic (fwd: read x, write y; bwd: read x and dy,
    write dx; the per-row statistics and per-feature parameters are left
    out) and the fraction of the measured copy peak."""
    out = {}
    peak, _ = load_peaks()
    stream = torch.cuda.current_stream()
    for w in synth.ROW_WORKLOADS:
        inp = synth.make_row_inputs(w, "cuda", seed=0)
        x, dy, gm, bt = inp["x"], inp["dy"], inp["gamma"], inp["beta"]
        y, dx = torch.empty_like(x), torch.empty_like(x)
        mean = torch.empty(w.M, device="cuda")
        rstd = torch.empty(w.M, device="cuda")
        dg = torch.empty(w.N, device="cuda")
        db = torch.empty(w.N, device="cuda")
        ws = torch.empty(max(gn.ln_workspace_size(w.M, w.N, w.dtype), 16), dtype=torch.uint8,
                         device="cuda")
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps + 3)]
        for ev in evs:
            flush()
            ev[0].record(stream)
            rc = (gn.ln_fwd_raw(x, w.M, w.N, gm, bt, w.eps, y, mean, rstd, stream) if w.op == "ln"
                  else gn.rms_fwd_raw(x, w.M, w.N, gm, w.eps, y, rstd, stream))
            ev[1].record(stream)
            assert rc == 0
            flush()
            ev[2].record(stream)
            rc = (gn.ln_bwd_raw(dy, x, mean, rstd, gm, w.M, w.N, dx, dg, db, ws, stream)
                  if w.op == "ln" else gn.rms_bwd_raw(dy, x, rstd, gm, w.M, w.N, dx, dg, ws, stream))
            ev[3].record(stream)
            assert rc == 0
        torch.cuda.synchronize()
        f = statistics.median(e[0].elapsed_time(e[1]) for e in evs[3:]) * 1e3
        b = statistics.median(e[2].elapsed_time(e[3]) for e in evs[3:]) * 1e3
        e_bytes = w.E * esize(w.dtype)
        fg, bg = 2 * e_bytes / (f * 1e-6) / 1e9, 3 * e_bytes / (b * 1e-6) / 1e9
        out[w.name] = {"fwd_us": round(f, 2), "bwd_us": round(b, 2), "fwd_gbs": round(fg, 1),
                       "bwd_gbs": round(bg, 1), "fwd_frac": round(fg / peak, 4),
                       "bwd_frac": round(bg / peak, 4),
                       "mi350x_bwd_us_context": ROW_MI350X_BWD_US.get(w.name)}
        del x, dy, y, dx, inp, ws
        torch.cuda.empty_cache()
    return out


def run_e2e(args, torch, dist, world, stream, x, dy, gm, bt, y, dx, mean, rstd, dg, db, fwd,
            bwd, flush, bytes_step):
    """The same metric through the C ABI with pinned host buffers: every step
    copies x, dy, gamma, beta in and y, dx, mean, rstd, dgamma, dbeta out.
    The host link moves about 210 GB/s each way here (copy engines and SM
    loads alike) and more with both directions busy, so the copies follow the
    op's data flow: an input stream brings gamma, beta and x, then dy; the
    forward starts once x has landed (dy arrives meanwhile); an output stream
    sends y, mean and rstd back while the backward runs; dx and the parameter
    gradients follow the backward.  All of it lies between the step's events."""
    w_numel = x.numel()
    hx = x.cpu().pin_memory()
    hdy = dy.cpu().pin_memory()
    hg, hb = gm.cpu().pin_memory(), bt.cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    hdx = torch.empty_like(hx).pin_memory()
    hmean, hrstd = mean.cpu().pin_memory(), rstd.cpu().pin_memory()
    hdg, hdb = dg.cpu().pin_memory(), db.cpu().pin_memory()
    h2d = (hx.numel() + hdy.numel()) * hx.element_size() + (hg.numel() + hb.numel()) * 4
    d2h = ((hy.numel() + hdx.numel()) * hy.element_size()
           + (hmean.numel() + hrstd.numel() + hdg.numel() + hdb.numel()) * 4)
    assert hx.numel() == w_numel
    s_in, s_out = torch.cuda.Stream(device=x.device), torch.cuda.Stream(device=x.device)
    Ke = max(3, min(10, args.steps))
    times = []
    for k in range(Ke + 2):
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        x_in, dy_in, f_done = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        a.record(stream)
        s_in.wait_stream(stream)
        with torch.cuda.stream(s_in):
            gm.copy_(hg, non_blocking=True)
            bt.copy_(hb, non_blocking=True)
            x.copy_(hx, non_blocking=True)
            x_in.record(s_in)
            dy.copy_(hdy, non_blocking=True)
            dy_in.record(s_in)
        stream.wait_event(x_in)
        fwd()
        f_done.record(stream)
        s_out.wait_event(f_done)
        with torch.cuda.stream(s_out):
            hy.copy_(y, non_blocking=True)
            hmean.copy_(mean, non_blocking=True)
            hrstd.copy_(rstd, non_blocking=True)
        stream.wait_event(dy_in)
        bwd()
        hdx.copy_(dx, non_blocking=True)
        hdg.copy_(dg, non_blocking=True)
        hdb.copy_(db, non_blocking=True)
        stream.wait_stream(s_out)
        b.record(stream)
        torch.cuda.synchronize()
        if k >= 2:
            times.append(a.elapsed_time(b))
        flush()
    ms = torch.tensor([statistics.mean(times)], dtype=torch.float64, device=x.device)
    if world > 1:
        dist.all_reduce(ms, op=dist.ReduceOp.MAX)
    value = world * bytes_step / (float(ms.item()) * 1e-3) / 1e9
    return {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(float(ms.item()), 3)}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from backward_normalization_gb300 import gn, replicas, synth

    gn.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    w = synth.BY_NAME[WORKLOAD]
    inp = synth.make_inputs(w, dev, seed=replicas.rank_seed(0, rank))
    x, dy, gm, bt = inp["x"], inp["dy"], inp["gamma"], inp["beta"]
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    mean = torch.empty(w.N * w.G, device=dev)
    rstd = torch.empty(w.N * w.G, device=dev)
    dg = torch.empty(w.C, device=dev)
    db = torch.empty(w.C, device=dev)
    ws = gn.alloc_workspace(gn.OP_BWD, w.N, w.C, w.HW, w.G, w.layout, x.dtype, dev)
    replicas.broadcast_params(gm, bt)  # one model: rank 0's gamma and beta everywhere
    grad_sum = replicas.ParamGradSum(w.C, dev)
    flush_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        # a read-only sweep over 4x the L2: evicts the workload's lines and
        # leaves clean ones, so no write-back lands in the next timed kernel
        torch.sum(flush_buf, dim=0, out=flush_out)

    def fwd():
        rc = gn.fwd_raw(x, w.N, w.C, w.HW, w.G, w.layout, gm, bt, w.eps, y, mean, rstd, ws, stream)
        if rc:
            raise RuntimeError(f"gn_fwd failed: {rc}")

    def bwd():
        rc = gn.bwd_raw(dy, x, mean, rstd, gm, w.N, w.C, w.HW, w.G, w.layout, dx, dg, db, ws, stream)
        if rc:
            raise RuntimeError(f"gn_bwd failed: {rc}")
        grad_sum(dg, db)  # dgamma/dbeta over all ranks, rank order (no-op on one rank)

    def step(evs=None):
        if evs:
            gn.set_timing_events(evs[0], evs[1], evs[2])
        fwd()
        if evs:
            gn.set_timing_events(evs[3], evs[4], evs[5])
        bwd()
        if evs:
            gn.set_timing_events()

    for _ in range(args.warmup):
        step()
        flush()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(K):
        # only the step's first and last events: an event between two kernels
        # would hold back the early launch of the second one
        step([evs[k][0], None, None, None, None, evs[k][5]])
        flush()  # L2 flushed between steps (outside the per-step event windows)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if rank == 0 else None
    per_step = [e[0].elapsed_time(e[5]) for e in evs]          # ms, fwd start -> bwd end

    # per-kernel durations: the same steps with an event between every two
    # kernels (each kernel then runs on its own)
    Ks = min(K, 50)
    for k in range(Ks):
        step(evs[k])
        flush()
    torch.cuda.synchronize()
    plan_f = gn.plan_info(0, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
    plan_b = gn.plan_info(1, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
    kb = kernel_bytes(w, plan_f.regime, plan_b.regime)
    kern = {}
    for e in evs[:Ks]:
        for k, v in kernel_times(kb, e).items():
            kern.setdefault(k, []).append(v)
    step_sum = torch.tensor([sum(per_step)], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(step_sum, op=dist.ReduceOp.MAX)
    ms_per_step = float(step_sum.item()) / K
    mb = min_bytes(w)
    bytes_step = mb["fwd"] + mb["bwd"]
    value = world * bytes_step / (ms_per_step * 1e-3) / 1e9

    # ---- e2e through the C ABI with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, torch, dist, world, stream, x, dy, gm, bt, y, dx, mean, rstd, dg, db,
                      fwd, bwd, flush, bytes_step)

    if rank != 0:
        return 0

    peak, peak_kind = load_peaks()
    totals = {k: sum(v) for k, v in kern.items()}
    dom = max(totals, key=totals.get)
    avg_ms = totals[dom] / Ks
    achieved = kb[dom] / (avg_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic_from_profiles(dom),
                "kernel": dom, "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": kb[dom], "avg_launch_us": round(avg_ms * 1e3, 2),
                "kernels": {k: {"avg_us": round(totals[k] / Ks * 1e3, 2),
                                "frac": round(kb[k] / (totals[k] / Ks * 1e-3) / 1e9 / peak, 4)}
                            for k in kb}}

    per_config = None
    if not args.no_per_config and world == 1:
        del x, dy, y, dx, inp
        torch.cuda.empty_cache()
        per_config = time_configs(gn, synth, torch, flush,
                                  names=args.configs.split(",") if args.configs else None,
                                  reps=args.reps, variants=not args.configs)

    rows = None
    if not args.no_per_config and not args.no_rows and world == 1:
        rows = time_rows(gn, synth, torch, flush, reps=args.reps)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        todo = synth.WORKLOADS[1:] if per_config is not None else [w]
        base = cpu_baselines(todo)
        b = base[w.name]
        cpu = {"value": b["all_cores_gbs"], "unit": UNIT, "cores": b["cores"], "kind": "oracle",
               "sample": b["sample"], "single_thread_value": b["single_thread_gbs"],
               "seconds": b["seconds_all_cores"]}
        for name, v in base.items():
            if per_config and name in per_config:
                per_config[name]["cpu_oracle"] = v

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_of(w, {
            "l2": "inputs larger than L2 (512 MiB per tensor); L2 also flushed between steps by a 512 MiB read",
            "parallelism": f"replicas x{world}, dgamma/dbeta summed across ranks",
            "frac_of_measured_peak": round(value / world / peak, 4),
            "frac_of_8tbs": round(value / world / 8000.0, 4)}),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (plan_f.launches + plan_b.launches) * K,
        "clocks": clk,
        "per_config": per_config,
        "rows_per_config": rows,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the LayerNorm / RMSNorm leg (rows_per_config)")
    ap.add_argument("--configs", default="",
                    help="comma-separated workload names for the per-workload leg; name:N overrides the batch")
    ap.add_argument("--reps", type=int, default=20, help="timed calls per workload in the per-workload leg")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    rc = run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())

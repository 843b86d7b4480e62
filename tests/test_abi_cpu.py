"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, validates arguments before touching the device, sizes
workspaces and plans consistently.  No compute call is made here."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from backward_normalization_gb300 import build as lib_build
from backward_normalization_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gn():
    lib_build.build()
    from backward_normalization_gb300 import gn as mod

    mod.lib()
    return mod


def _declared_symbols():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"GN_API[^;{(]*?\b(\w+)\s*\(", txt)
    return sorted(n for n in set(names) if not n.startswith("__"))  # not the macro itself


def test_every_declared_symbol_is_exported(gn):
    names = _declared_symbols()
    assert "gn_fwd" in names and "gn_bwd" in names and "gn_workspace_size" in names
    L = gn.lib()
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_status_strings(gn):
    for s in range(6):
        assert gn.status_string(s).startswith("GN_")
    assert "unknown" in gn.status_string(99)


def test_workspace_size(gn):
    for w in synth.WORKLOADS:
        for op in (0, 1):
            n = gn.workspace_size(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
            assert n > 0 and n % 256 == 0
            d = gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype, aligned=True)
            assert d.workspace_bytes <= n
            d1 = gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype, aligned=False)
            assert d1.workspace_bytes <= n
    # invalid or empty problems need no workspace
    assert gn.workspace_size(0, 2, 6, 4, 4, "nchw", "f32") == 0   # G does not divide C
    assert gn.workspace_size(0, 0, 8, 4, 2, "nhwc", "f16") == 0
    assert gn.workspace_size(1, 2, 8, 0, 2, "nhwc", "f16") == 0
    assert gn.workspace_size(7, 2, 8, 4, 2, "nhwc", "f16") == 0
    assert gn.lib().gn_workspace_size(0, 2, 8, 4, 2, 5, 0) == 0


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced


def _fwd(gn, **kw):
    a = dict(x=FAKE, N=2, C=8, HW=16, G=2, layout=0, dtype=0, gamma=None, beta=None, eps=1e-5,
             y=FAKE * 2, mean=FAKE * 3, rstd=FAKE * 4, ws=FAKE * 5, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return gn.lib().gn_fwd(a["x"], a["N"], a["C"], a["HW"], a["G"], a["layout"], a["dtype"],
                           a["gamma"], a["beta"], a["eps"], a["y"], a["mean"], a["rstd"], a["ws"],
                           a["ws_bytes"], a["stream"])


def _bwd(gn, **kw):
    a = dict(dy=FAKE, x=FAKE * 2, mean=FAKE * 3, rstd=FAKE * 4, gamma=None, N=2, C=8, HW=16, G=2,
             layout=1, dtype=1, dx=FAKE * 5, dgamma=None, dbeta=None, ws=FAKE * 6,
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return gn.lib().gn_bwd(a["dy"], a["x"], a["mean"], a["rstd"], a["gamma"], a["N"], a["C"],
                           a["HW"], a["G"], a["layout"], a["dtype"], a["dx"], a["dgamma"],
                           a["dbeta"], a["ws"], a["ws_bytes"], a["stream"])


def test_validation_before_any_launch(gn):
    INV, UNS, WS = gn.GN_ERR_INVALID, gn.GN_ERR_UNSUPPORTED, gn.GN_ERR_WORKSPACE
    assert _fwd(gn, G=3) == INV                 # 3 does not divide 8
    assert _fwd(gn, G=0) == INV
    assert _fwd(gn, N=-1) == INV
    assert _fwd(gn, layout=2) == UNS
    assert _fwd(gn, dtype=5) == UNS
    assert _fwd(gn, x=None) == INV
    assert _fwd(gn, mean=None) == INV
    assert _fwd(gn, eps=-1.0) == INV
    assert _fwd(gn, eps=float("nan")) == INV
    assert _fwd(gn, y=FAKE + 4) == INV           # y overlaps x without being x
    assert _fwd(gn, mean=FAKE + 8) == INV        # stats inside x
    assert _fwd(gn, ws=None) == WS
    assert _fwd(gn, ws_bytes=8) == WS
    assert _fwd(gn, ws=FAKE * 5 + 8) == WS       # misaligned workspace
    assert _fwd(gn, N=0) == 0                    # empty: nothing to do
    assert _fwd(gn, HW=0, x=None) == 0
    assert _bwd(gn, G=5) == INV
    assert _bwd(gn, dy=None) == INV
    assert _bwd(gn, dx=FAKE * 2 + 2) == INV      # dx overlaps x without being x
    assert _bwd(gn, dgamma=FAKE * 7, dbeta=FAKE * 7) == INV
    assert _bwd(gn, ws_bytes=0) == WS
    assert _bwd(gn, C=0) == 0
    need = gn.plan_info(1, 2, 8, 16, 2, "nhwc", "f16", aligned=True).workspace_bytes
    assert need <= gn.workspace_size(1, 2, 8, 16, 2, "nhwc", "f16")
    assert _bwd(gn, ws_bytes=need - 1) == WS


def test_row_length_limit_independent_of_problem_size(gn):
    """LayerNorm / RMSNorm forward rows up to 256 threads x 32 values (8192
    values, fp32 too) are planned whatever the row count (small problems take
    fewer values per thread only where the row still fits a team); the
    backward takes rows up to 256 x 16 values (4096); longer rows give
    GN_ERR_UNSUPPORTED.  Checked on the host: without a device a planned call
    goes on to its launch and fails there (GN_ERR_CUDA), an unplannable one
    is refused before."""
    L = gn.lib()
    x, y, mean, rstd = 1 << 40, 2 << 40, 3 << 40, (3 << 40) + (1 << 32)
    dx, dy, ws = 4 << 40, 5 << 40, 6 << 40

    def fwd(M, N, dt, rms=False):
        if rms:
            return L.rms_fwd(x, M, N, dt, None, 1e-5, y, rstd, None)
        return L.ln_fwd(x, M, N, dt, None, None, 1e-5, y, mean, rstd, None)

    def bwd(M, N, dt):
        return L.ln_bwd(dy, x, mean, rstd, None, M, N, dt, dx, None, None, ws, 1 << 30, None)

    UNS = gn.GN_ERR_UNSUPPORTED
    for M in (1, 64, 2048, 131072):
        for dt in (1, 2):  # fp16, bf16
            assert fwd(M, 8192, dt) != UNS and fwd(M, 8192, dt, rms=True) != UNS
            assert fwd(M, 4096, dt) != UNS and fwd(M, 16384, dt) == UNS
            assert bwd(M, 4096, dt) != UNS and bwd(M, 8192, dt) == UNS
        assert fwd(M, 8192, 0) != UNS and fwd(M, 16384, 0) == UNS  # fp32
        assert bwd(M, 4096, 0) != UNS and bwd(M, 8192, 0) == UNS


def test_plan_vector_width_and_modes(gn):
    d = gn.plan_info(0, 1, 128, 2048 * 1024, 16, "nhwc", "f16")
    assert d.vector_width == 8 and d.launches == 3  # workspace clear + two kernels
    assert gn.plan_info(0, 2, 6, 77, 3, "nhwc", "f16").vector_width == 1       # C*2 % 16 != 0
    assert gn.plan_info(0, 2, 64, 2303, 8, "nchw", "f32").vector_width == 1    # HW*4 % 16 != 0
    assert gn.plan_info(0, 2, 64, 2304, 8, "nchw", "f32").vector_width == 4
    gn.set_regime(gn.REGIME_TWO_KERNEL)
    try:
        # two-kernel path: small planes get a warp each, large planes a CTA per chunk
        assert gn.plan_info(0, 2, 32, 256, 8, "nchw", "f32").threads == 256
        assert gn.plan_info(0, 2, 64, 4096, 8, "nchw", "f32").threads == 512
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    for w in synth.WORKLOADS:
        d = gn.plan_info(1, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
        assert 0 < d.ctas < 2 ** 31
        assert d.threads % 32 == 0 or w.layout == "nhwc"


def test_regime_choice(gn):
    # the 512 MiB single-sample workload is too large for a cluster to hold
    assert gn.plan_info(0, 1, 128, 2048 * 1024, 16, "nhwc", "f16").regime == 0
    # misaligned inputs (scalar path) always take the two-kernel path
    assert gn.plan_info(0, 2, 64, 2304, 8, "nchw", "f32", aligned=False).regime == 0
    gn.set_regime(gn.REGIME_TWO_KERNEL)
    try:
        d = gn.plan_info(1, 8, 320, 4096, 32, "nhwc", "bf16")
        assert d.regime == 0 and d.launches == 3
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    gn.set_regime(gn.REGIME_RESIDENT)
    try:
        d = gn.plan_info(1, 8, 320, 4096, 32, "nhwc", "bf16")
        assert d.regime == 1 and d.launches == 2
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    # the wave kernel clears its own counters: one launch per op
    gn.set_regime(gn.REGIME_WAVE)
    try:
        d = gn.plan_info(1, 8, 320, 4096, 32, "nhwc", "bf16")
        assert d.regime == 3 and d.launches == 1
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    gn.set_regime(gn.REGIME_FLAT)
    try:
        d = gn.plan_info(1, 8, 320, 4096, 32, "nhwc", "bf16")
        assert d.regime == 4 and d.launches == 1
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    with pytest.raises(gn.GnError):
        gn.set_regime(7)


def test_finalisation_placement(gn):
    """NCHW two-kernel plans finalise in the second kernel when each of its
    CTAs reads at most 4 KB of partial records; otherwise (and always for
    channels-last) the first kernel's last arrival of a sample does it, after
    level-1 merges of 8 items when a sample has 16 items or more."""
    gn.set_regime(gn.REGIME_TWO_KERNEL)
    try:
        # NCHW planes: one group's Cg records per CTA
        d = gn.plan_info(1, 112, 64, 512 * 512, 8, "nchw", "f32")
        assert (d.finalise_second, d.level1_items) == (1, 1)
        # NCHW small planes (blocks of rows)
        d = gn.plan_info(0, 2, 36, 100, 3, "nchw", "f32")
        assert (d.finalise_second, d.level1_items) == (1, 1)
        # channels-last keeps the chain even with few records
        d = gn.plan_info(1, 16, 32, 64, 8, "nhwc", "bf16")
        assert (d.finalise_second, d.level1_items) == (0, 1)
        # one sample, 128 channels, hundreds of items: the chain, with level-1 merges
        d = gn.plan_info(0, 1, 128, 2048 * 1024, 16, "nhwc", "f16")
        assert (d.finalise_second, d.level1_items) == (0, 8)
        # 512 channels, a few items per sample: the chain
        d = gn.plan_info(1, 32, 512, 32 * 32, 32, "nhwc", "bf16")
        assert (d.finalise_second, d.level1_items) == (0, 1)
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    # the resident regime finalises in its one kernel
    gn.set_regime(gn.REGIME_RESIDENT)
    try:
        d = gn.plan_info(0, 8, 320, 4096, 32, "nhwc", "bf16")
        assert d.regime == 1 and d.finalise_second == 0
    finally:
        gn.set_regime(gn.REGIME_AUTO)


def test_f64_storage_plans(gn):
    """fp64 is accepted as a storage type: 16-byte vectors of two doubles, or
    the scalar path, always on the two-kernel path (whatever regime is
    asked for); the row family does not take it."""
    d = gn.plan_info(0, 2, 16, 4096, 4, "nchw", "f64")
    assert (d.regime, d.vector_width, d.launches) == (0, 2, 3)
    assert gn.plan_info(1, 3, 40, 99, 8, "nhwc", "f64").vector_width == 2
    assert gn.plan_info(1, 2, 3, 25, 3, "nhwc", "f64").vector_width == 1   # 3 doubles: not 16 B
    assert gn.plan_info(0, 2, 6, 63, 3, "nchw", "f64").vector_width == 1   # 63 doubles per plane
    for reg in (gn.REGIME_RESIDENT, gn.REGIME_PIPELINED, gn.REGIME_WAVE, gn.REGIME_FLAT):
        gn.set_regime(reg)
        try:
            assert gn.plan_info(1, 2, 16, 4096, 4, "nchw", "f64").regime == 0
            assert gn.plan_info(0, 8, 64, 1024, 8, "nhwc", "f64").regime == 0
        finally:
            gn.set_regime(gn.REGIME_AUTO)
    # workspace of an f64 problem: the same records as the fp32 one
    assert gn.lib().gn_workspace_size(1, 2, 16, 4096, 4, 0, 3) > 0
    assert gn.lib().ln_workspace_size(16, 64, 3) == 0


def test_automatic_choice(gn):
    """The automatic choice: the wave regime for NCHW problems of at least
    32 MiB with units of at least 64 KiB; the flat regime for channels-last
    backwards of 10-48 MiB (x and dy); the resident regime for channels-last
    forwards and small NCHW units when one wave of clusters covers every unit
    (or the input is tiny); the two-kernel path otherwise."""
    assert gn.plan_info(1, 112, 64, 512 * 512, 8, "nchw", "f32").regime == 3   # 8 MiB units
    assert gn.plan_info(0, 112, 64, 512 * 512, 8, "nchw", "f32").regime == 3
    assert gn.plan_info(0, 16, 64, 512 * 512, 64, "nchw", "f32").regime == 3   # 1 MiB units
    assert gn.plan_info(1, 256, 64, 64 * 64, 8, "nchw", "f32").regime == 3     # 128 KiB units
    assert gn.plan_info(1, 4, 64, 64 * 64, 8, "nchw", "f32").regime != 3       # 4 MiB input
    assert gn.plan_info(0, 2, 32, 256, 8, "nchw", "f32").regime == 1        # 64 KB
    assert gn.plan_info(0, 512, 32, 256, 8, "nchw", "f32").regime == 0      # 4096 units
    assert gn.plan_info(0, 8, 320, 4096, 32, "nhwc", "bf16").regime == 1    # 32 clusters
    assert gn.plan_info(0, 64, 320, 4096, 32, "nhwc", "bf16").regime == 0   # 256 clusters
    assert gn.plan_info(1, 8, 320, 4096, 32, "nhwc", "bf16").regime == 4   # 40 MiB backward
    assert gn.plan_info(1, 2, 320, 4096, 32, "nhwc", "bf16").regime == 4   # 10 MiB
    assert gn.plan_info(1, 32, 512, 1024, 32, "nhwc", "bf16").regime == 0  # 64 MiB
    assert gn.plan_info(1, 1, 320, 4096, 32, "nhwc", "bf16").regime != 4   # 5 MiB
    assert gn.plan_info(1, 8, 320, 4096, 32, "nhwc", "bf16", aligned=False).regime == 0
    assert gn.plan_info(0, 1, 128, 2048 * 1024, 16, "nhwc", "f16").regime == 0
    assert gn.plan_info(0, 2, 64, 2303, 8, "nchw", "f32").regime == 0       # scalar path
    assert gn.plan_info(1, 2, 16, 4096 * 256, 4, "nchw", "f64").regime == 0  # f64 storage
    gn.set_regime(gn.REGIME_RESIDENT)  # asked for: wherever the problem fits
    try:
        assert gn.plan_info(0, 512, 32, 256, 8, "nchw", "f32").regime == 1
    finally:
        gn.set_regime(gn.REGIME_AUTO)


def test_wave_plans(gn):
    """Wave plans: a unit's pieces all fit on co-resident CTAs (P <= CTAs),
    pieces hold whole 16-byte vectors and wait in tensor memory, and one CTA
    holds each SM.  (A unit may straddle two steps: with the pieces held in
    tensor memory that measured no slower.)"""
    gn.set_regime(gn.REGIME_WAVE)
    try:
        plans = [(w, gn.plan_info(op, w.N, w.C, w.HW, w.G, w.layout, w.dtype))
                 for w in synth.WORKLOADS[2:] for op in (0, 1)]
    finally:
        gn.set_regime(gn.REGIME_AUTO)
    for w, d in plans:
        assert d.regime == 3 and d.launches == 1
        assert d.hold_buffers >= 2 and d.slots >= 2  # pieces wait in tensor memory
        assert d.smem_bytes > 114 * 1024  # one tensor-memory holder per SM
        assert 1 <= d.pieces_per_unit <= d.ctas
        assert d.smem_bytes <= 227 * 1024
        if w.layout == "nchw":
            assert d.piece_elems * (4 if w.dtype == "f32" else 2) % 16 == 0
    gn.set_regime(gn.REGIME_WAVE)
    try:
        assert gn.plan_info(0, 1, 128, 2048 * 1024, 16, "nhwc", "f16").regime == 0  # too large
    finally:
        gn.set_regime(gn.REGIME_AUTO)


def test_flat_plans(gn):
    """Flat plans: one CTA per SM (at most one per row), one launch (no
    separate workspace clear), whole row vectors per thread, and a forward
    that holds each CTA's whole run in shared memory when it fits; only
    dense, 16-byte aligned channels-last fp32 / fp16 / bf16 problems take it."""
    gn.set_regime(gn.REGIME_FLAT)
    try:
        for N, C, HW, G, dt in ((8, 320, 4096, 32, "bf16"), (32, 512, 1024, 32, "bf16"),
                                (4, 512, 16384, 32, "bf16"), (2, 64, 300, 8, "f32")):
            for op in (0, 1):
                d = gn.plan_info(op, N, C, HW, G, "nhwc", dt)
                esz = 4 if dt == "f32" else 2
                assert (d.regime, d.launches, d.ctas) == (4, 1, min(152, N * HW))
                assert d.threads % (C * esz // 16) == 0 and d.threads <= 512
                assert 1 <= d.slots <= 32 and d.smem_bytes <= 227 * 1024
                # a chunk's copy (x, and dy) completes one mbarrier phase
                assert d.piece_elems * C * esz * (1 + op) < 1 << 20
        # c4's forward run (216 rows of 1 KiB) stays in shared memory: as many
        # slots as chunks
        d = gn.plan_info(0, 32, 512, 1024, 32, "nhwc", "bf16")
        assert d.slots == d.pieces_per_unit
        assert gn.plan_info(0, 7, 16, 1, 4, "nhwc", "bf16").ctas == 7  # one row per CTA
        assert gn.plan_info(0, 2, 64, 2304, 8, "nchw", "f32").regime == 0
        assert gn.plan_info(0, 2, 40, 99, 8, "nhwc", "f64").regime == 0
        assert gn.plan_info(0, 2, 40, 99, 8, "nhwc", "f32", aligned=False).regime == 0
        assert gn.plan_info(0, 3, 6, 77, 3, "nhwc", "f16").regime == 0   # rows not 16-byte vectors
        assert gn.plan_info(1, 2, 4096, 40, 32, "nhwc", "f16").regime == 0  # 512 columns: scratch too large
    finally:
        gn.set_regime(gn.REGIME_AUTO)


def test_configs_cover_both_layouts_and_vector_paths(gn):
    seen = set()
    for w in synth.WORKLOADS:
        d = gn.plan_info(0, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
        seen.add((w.layout, d.vector_width > 1, d.threads))
    assert {s[0] for s in seen} == {"nchw", "nhwc"}


def test_workspace_layout_error_word_first(gn):
    """The error word sits at offset 0 and the counters after it; each call
    clears that prefix itself, the same for both ops of a problem."""
    for w in synth.WORKLOADS:
        f = gn.plan_info(0, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
        b = gn.plan_info(1, w.N, w.C, w.HW, w.G, w.layout, w.dtype)
        assert f.err_offset == 0 and b.err_offset == 0
        assert f.clear_bytes == b.clear_bytes
        assert 20 <= f.clear_bytes <= gn.workspace_size(0, w.N, w.C, w.HW, w.G, w.layout, w.dtype)


def test_workspace_status_rejects_bad_workspace(gn):
    assert gn.lib().gn_workspace_status(None, None) == gn.GN_ERR_WORKSPACE
    assert gn.lib().gn_workspace_status(FAKE + 4, None) == gn.GN_ERR_WORKSPACE


def test_fault_injection_launch(gn):
    """GN_FAULT_LAUNCH: a valid call fails with GN_ERR_CUDA before anything
    is enqueued (nothing touches the fake pointers), invalid calls are still
    reported as invalid, and clearing the mode restores normal validation."""
    gn.set_fault_injection(gn.FAULT_LAUNCH)
    try:
        assert _fwd(gn) == gn.GN_ERR_CUDA
        assert gn.lib().gn_last_cuda_error() == 719  # cudaErrorLaunchFailure
        assert _bwd(gn) == gn.GN_ERR_CUDA
        assert _bwd(gn, HW=0, dgamma=FAKE * 7, dbeta=FAKE * 8) == gn.GN_ERR_CUDA
        assert _fwd(gn, G=3) == gn.GN_ERR_INVALID
        assert _fwd(gn, ws_bytes=8) == gn.GN_ERR_WORKSPACE
        assert _fwd(gn, N=0) == 0
    finally:
        gn.set_fault_injection(gn.FAULT_NONE)
    with pytest.raises(gn.GnError):
        gn.set_fault_injection(9)


def test_fault_injection_from_environment(gn):
    """GN_FAULT_INJECT=launch in the environment of a fresh process."""
    import subprocess
    import sys

    code = ("import sys; sys.path.insert(0, %r)\n"
            "from backward_normalization_gb300 import gn\n"
            "F = 1 << 20\n"
            "rc = gn.lib().gn_fwd(F, 2, 8, 16, 2, 0, 0, None, None, 1e-5, F * 2, F * 3, F * 4,"
            " F * 5, 1 << 30, None)\n"
            "print(rc, gn.lib().gn_last_cuda_error())\n") % ROOT
    env = dict(os.environ, GN_FAULT_INJECT="launch")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr
    rc, err = map(int, out.stdout.split())
    assert rc == gn.GN_ERR_CUDA and err == 719


def _fwd_ex(gn, **kw):
    a = dict(x=FAKE, xs=(8 * 16, 16), N=2, C=8, HW=16, G=2, layout=0, dtype=0, y=FAKE * 4,
             ys=(8 * 16, 16), mean=FAKE * 8, rstd=FAKE * 9, ws=FAKE * 10, ws_bytes=1 << 30)
    a.update(kw)
    return gn.lib().gn_fwd_ex(a["x"], a["xs"][0], a["xs"][1], a["N"], a["C"], a["HW"], a["G"],
                              a["layout"], a["dtype"], None, None, 1e-5, a["y"], a["ys"][0],
                              a["ys"][1], a["mean"], a["rstd"], a["ws"], a["ws_bytes"], None)


def test_strided_view_validation(gn):
    """gn_fwd_ex checks its strides before anything else happens; calls that
    pass validation run into GN_FAULT_LAUNCH here, so nothing is launched."""
    INV, CUDA = gn.GN_ERR_INVALID, gn.GN_ERR_CUDA
    gn.set_fault_injection(gn.FAULT_LAUNCH)
    try:
        assert _fwd_ex(gn) == CUDA                                   # dense NCHW
        assert _fwd_ex(gn, xs=(12 * 16, 16)) == CUDA                 # a channel slice of 12
        assert _fwd_ex(gn, xs=(16, 2 * 16)) == CUDA                  # channel-major batch
        assert _fwd_ex(gn, xs=(8 * 20, 20)) == CUDA                  # padded planes
        assert _fwd_ex(gn, xs=(8 * 16, 15)) == INV                   # planes overlap
        assert _fwd_ex(gn, xs=(7 * 16, 16)) == INV                   # samples overlap
        assert _fwd_ex(gn, xs=(-128, 16)) == INV
        assert _fwd_ex(gn, N=1, xs=(5, 16)) == CUDA                  # N = 1: sample stride free
        nhwc = dict(layout=1, ys=(16 * 8, 8))
        assert _fwd_ex(gn, xs=(16 * 8, 8), **nhwc) == CUDA           # dense NHWC
        assert _fwd_ex(gn, xs=(16 * 10, 10), **nhwc) == CUDA         # channel slice, NHWC
        assert _fwd_ex(gn, xs=(16 * 8, 7), **nhwc) == INV            # rows overlap
        # an output whose span meets the input's is rejected unless it is the input in place
        assert _fwd_ex(gn, y=FAKE + 64) == INV
        assert _fwd_ex(gn, y=FAKE) == CUDA
        assert _fwd_ex(gn, y=FAKE, ys=(8 * 20, 20)) == INV
    finally:
        gn.set_fault_injection(gn.FAULT_NONE)

"""Flat-regime plans, checked on the host (no GPU): the row runs, chunks,
segments, record slots and owner shares that gn_flat.cu walks, re-derived here
from the plan the library reports, for shapes whose runs cut samples at odd
rows, hold several samples, or stream through a ring.

For every CTA b of a plan (runs [b*R/NB, (b+1)*R/NB), R = N*HW):
  * pass 1 walks chunks 0..nk-1 and, inside each, the pieces between segment
    boundaries: every row is folded exactly once, in the segment it belongs
    to, and the segments end (their records are written) in order;
  * pass 2 walks the chunks in reverse, each from the slot that holds it
    (the last S chunks stay from pass 1, the others are copied in again after
    the chunk S places later has been written out): every row once again;
  * the merge reads, for each sample, the records (CTA, segment) of the CTAs
    whose runs touch it -- each of them written by pass 1;
  * owner shares [b*NP/NB, (b+1)*NP/NB) cover every pair (forward: N*G) or
    item (backward: N*C) exactly once;
and the records fit in the workspace the library asks for.
"""
from __future__ import annotations

import pytest

from backward_normalization_gb300 import gn

SHAPES = [
    (8, 320, 4096, 32, "bf16"), (32, 512, 1024, 32, "bf16"), (32, 512, 1024, 512, "bf16"),
    (2, 320, 1024, 32, "bf16"), (3, 320, 289, 32, "bf16"), (2, 48, 50, 48, "bf16"),
    (7, 16, 1, 4, "bf16"), (2, 64, 300, 8, "f32"), (1, 32, 90000, 8, "bf16"),
    (40, 64, 2304, 8, "bf16"), (2, 1200, 6, 15, "f32"), (300, 64, 2, 8, "bf16"),
    (64, 64, 9, 8, "f16"), (4, 512, 16384, 32, "bf16"), (8, 320, 1536, 32, "f16"),
    (16, 256, 576, 16, "f32"), (1000, 8, 3, 2, "bf16"), (152, 16, 1, 2, "bf16"),
    (153, 16, 1, 2, "bf16"), (2, 40, 99, 8, "f32"),
]
ESZ = {"f32": 4, "f16": 2, "bf16": 2}


def cdiv(a, b):
    return (a + b - 1) // b


@pytest.fixture
def flat():
    gn.set_regime(gn.REGIME_FLAT)
    yield
    gn.set_regime(gn.REGIME_AUTO)


def _walk(N, C, HW, G, dtype, op):
    d = gn.plan_info(op, N, C, HW, G, "nhwc", dtype)
    assert d.regime == gn.REGIME_FLAT
    NB, S, chunk = d.ctas, d.slots, d.piece_elems
    R = N * HW
    assert NB == min(152, R)  # one CTA per SM (the host sizes plans for 152 without a device)
    esz = ESZ[dtype]
    assert chunk * C * esz * (1 + op) < 1 << 20  # one mbarrier phase's byte count
    assert 1 <= S <= 32 and d.smem_bytes <= 227 * 1024
    start = lambda b: b * R // NB
    run_of = lambda r: ((r + 1) * NB - 1) // R
    segmax = max((start(b + 1) - 1) // HW - start(b) // HW + 1 for b in range(NB))
    written = set()
    for b in range(NB):
        rA, rB = start(b), start(b + 1)
        nrows = rB - rA
        assert nrows >= 1 and run_of(rA) == b and run_of(rB - 1) == b
        nk = cdiv(nrows, chunk)
        nA = rA // HW
        nseg = (rB - 1) // HW - nA + 1
        assert nk <= d.pieces_per_unit
        seg_begin = lambda s: max(0, (nA + s) * HW - rA)
        seg_end = lambda s: min(nrows, (nA + s + 1) * HW - rA)
        # pass 1
        seen = [0] * nrows
        s, send, ended = 0, seg_end(0), []
        for k in range(nk):
            k0, k1 = k * chunk, min(nrows, (k + 1) * chunk)
            i0 = k0
            while i0 < k1:
                i1 = min(send, k1)
                for i in range(i0, i1):
                    seen[i] += 1
                    assert seg_begin(s) <= i < seg_end(s)
                if i1 == send:
                    ended.append(s)
                    written.add((b, s))
                    s += 1
                    if s < nseg:
                        send = seg_end(s)
                i0 = i1
        assert seen == [1] * nrows and ended == list(range(nseg))
        # pass 2
        slot = {k % S: k for k in range(nk)}
        seen = [0] * nrows
        s = nseg - 1
        sbeg = seg_begin(s)
        for k in range(nk - 1, -1, -1):
            assert slot[k % S] == k
            k0, i1 = k * chunk, min(nrows, (k + 1) * chunk)
            while True:
                i0 = max(sbeg, k0)
                for i in range(i0, i1):
                    seen[i] += 1
                    assert seg_begin(s) <= i < seg_end(s)
                if i0 == k0:
                    break
                s -= 1
                assert s >= 0
                sbeg, i1 = seg_begin(s), i0
            if k - S >= 0:
                slot[k % S] = k - S
        assert seen == [1] * nrows
    # the merge's reads
    for n in range(N):
        for bb in range(run_of(n * HW), run_of((n + 1) * HW - 1) + 1):
            assert (bb, n - start(bb) // HW) in written
    # owner shares
    NP = N * (C if op else G)
    owned = [0] * NP
    for b in range(NB):
        for P in range(b * NP // NB, (b + 1) * NP // NB):
            owned[P] += 1
    assert owned == [1] * NP
    # records fit in the workspace (its partial-sum region starts past the
    # error word and counters)
    recs = NB * segmax * (C if op else G)
    assert recs * 8 < d.workspace_bytes
    return d


@pytest.mark.parametrize("shape", SHAPES, ids=["x".join(map(str, s)) for s in SHAPES])
@pytest.mark.parametrize("op", [0, 1], ids=["fwd", "bwd"])
def test_flat_plan_walk(flat, shape, op):
    N, C, HW, G, dtype = shape
    if C * ESZ[dtype] // 16 > 512 or (C * ESZ[dtype]) % 16:
        pytest.skip("not a flat-regime shape")
    d = gn.plan_info(op, N, C, HW, G, "nhwc", dtype)
    if d.regime != gn.REGIME_FLAT:
        # declined only where its scratch or tables do not fit shared memory
        assert op == 1 or G * 8 > 32 << 10
        return
    _walk(N, C, HW, G, dtype, op)

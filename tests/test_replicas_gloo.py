"""Two data-parallel ranks on CPU (gloo): each rank takes its own seeded shard,
its parameter gradients come from the oracle (standing in for gn_bwd on its
GPU), and ParamGradSum combines them; broadcast_params gives every rank
rank 0's gamma.  The totals must be bit-identical on
both ranks, equal the rank-order float32 sum exactly, and match the oracle's
dgamma/dbeta of the whole batch (both shards as one batch)."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from backward_normalization_gb300 import replicas, synth

WORLD = 2
CASES = [synth.WORKLOADS[0], synth.WORKLOADS[2].scaled(name="r2", N=2, H=5, W=7)]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard(w, rank):
    inp = synth.make_inputs(w, "cpu", seed=replicas.rank_seed(0, rank))
    return {k: v.double().numpy() for k, v in inp.items()}


def _worker(rank, port, outdir, case):
    import oracle

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=WORLD)
    try:
        w = CASES[case]
        s = _shard(w, rank)
        _, dg, db = oracle.get().backward(s["dy"], s["x"], w.N, w.C, w.HW, w.G,
                                          synth.LAYOUTS[w.layout], s["gamma"], w.eps)
        dg_t = torch.tensor(dg, dtype=torch.float32)
        db_t = torch.tensor(db, dtype=torch.float32)
        np.save(os.path.join(outdir, f"own{rank}.npy"), np.concatenate([dg_t.numpy(), db_t.numpy()]))
        gm = torch.tensor(s["gamma"], dtype=torch.float32)
        replicas.broadcast_params(gm)
        np.save(os.path.join(outdir, f"gamma{rank}.npy"), gm.numpy())
        replicas.ParamGradSum(w.C, "cpu")(dg_t, db_t)
        np.save(os.path.join(outdir, f"tot{rank}.npy"), np.concatenate([dg_t.numpy(), db_t.numpy()]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", range(len(CASES)), ids=[w.name for w in CASES])
def test_two_ranks_sum_parameter_gradients(case, tmp_path):
    import oracle

    mp.start_processes(_worker, args=(_free_port(), str(tmp_path), case), nprocs=WORLD,
                       join=True, start_method="spawn")
    tot = [np.load(tmp_path / f"tot{r}.npy") for r in range(WORLD)]
    own = [np.load(tmp_path / f"own{r}.npy") for r in range(WORLD)]
    assert np.array_equal(tot[0], tot[1])                   # identical on every rank
    assert np.array_equal(tot[0], own[0] + own[1])          # rank order, float32
    g0 = np.float32(_shard(CASES[case], 0)["gamma"])
    assert all(np.array_equal(np.load(tmp_path / f"gamma{r}.npy"), g0) for r in range(WORLD))
    # the whole batch at once: the shards' samples one after the other
    w = CASES[case]
    sh = [_shard(w, r) for r in range(WORLD)]
    cat = {k: np.concatenate([s[k] for s in sh]) for k in ("x", "dy")}
    _, dg, db = oracle.get().backward(cat["dy"], cat["x"], WORLD * w.N, w.C, w.HW, w.G,
                                      synth.LAYOUTS[w.layout], sh[0]["gamma"], w.eps)
    ref = np.concatenate([dg, db])
    assert np.allclose(tot[0], ref, rtol=1e-5, atol=1e-5 * np.abs(ref).max())


def test_single_process_is_a_no_op():
    dg = torch.arange(4, dtype=torch.float32)
    db = torch.ones(4)
    replicas.ParamGradSum(4, "cpu")(dg, db)
    assert dg.tolist() == [0, 1, 2, 3] and db.tolist() == [1, 1, 1, 1]

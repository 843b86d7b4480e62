"""Data-parallel replicas of the GroupNorm step, one process per GPU.

GroupNorm's statistics are per sample, so a batch split across ranks needs no
exchange for y, mean, rstd or dx: each rank runs the forward and backward on
its own samples.  The only cross-rank quantity is the parameter gradient of
gamma and beta, which sums over the whole batch (the backward section of the
Group Normalization paper: dgamma and dbeta are sums over every sample and
position of the channel).  Each rank's gn_bwd gives the sum over its own
samples; ParamGradSum adds the ranks' vectors in rank order, so every rank
ends with bit-identical totals whatever the arrival order of the messages.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of a rank's synthetic shard (distinct per rank, fixed per run)."""
    return base_seed + rank


def broadcast_params(*tensors, src: int = 0, group=None) -> None:
    """Gives every rank rank `src`'s parameter values (replicas of one model
    share gamma and beta); nothing to do with one rank."""
    if not dist.is_initialized() or dist.get_world_size(group) == 1:
        return
    for t in tensors:
        dist.broadcast(t, src, group=group)


def rank_order_sum(parts):
    """parts[0] + parts[1] + ... in that order (fp32): the fixed order that
    makes every rank's totals bit-identical."""
    tot = parts[0].clone()
    for t in parts[1:]:
        tot += t
    return tot


class ParamGradSum:
    """Sums dgamma and dbeta over the ranks of a process group, in rank order.

    One all_gather of the concatenated [dgamma, dbeta] (2*C floats per rank),
    then rank 0's vector plus rank 1's plus ... on every rank.  With one rank
    it does nothing.
    """

    def __init__(self, C: int, device, group=None):
        self.C = C
        self.group = group
        self.world = dist.get_world_size(group) if dist.is_initialized() else 1
        self.parts = [torch.empty(2 * C, dtype=torch.float32, device=device)
                      for _ in range(self.world)]

    def __call__(self, dgamma: torch.Tensor, dbeta: torch.Tensor) -> None:
        if self.world == 1:
            return
        mine = torch.cat([dgamma.reshape(-1), dbeta.reshape(-1)])
        dist.all_gather(self.parts, mine, group=self.group)
        tot = rank_order_sum(self.parts)
        dgamma.copy_(tot[:self.C].view_as(dgamma))
        dbeta.copy_(tot[self.C:].view_as(dbeta))

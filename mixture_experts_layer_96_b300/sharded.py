"""The one exchange step of a layer whose batch is split by tokens over ranks.

Every unit's routing and expert FFN are local to the rank that holds it; only two things are
global over the batch ["第 10 课：专家并行 EP", §4: capacity C = CF·K·T/E, overflow tokens
dropped in arrival order; L_aux = α·E·Σ_i f_i·P_i with f_i and P_i over the whole batch]:

  - an expert's queue runs over the whole batch in token order, so rank r's picks of expert e
    start at the picks of e on ranks 0..r-1: an exclusive scan over ranks of the E pre-drop
    counts (all-gather of E int32 per rank), fed to moe_dispatch_sharded with the batch's size;
  - the aux loss needs the batch's per-expert pick counts and Σ_t p_{t,e}: an all-reduce of 2E
    values.

Ranks hold consecutive token ranges in rank order. The collectives are torch.distributed's (NCCL on
GPUs, gloo on CPU); around them there is only a sum over ranks of E counts and the aux loss's
2E-term formula. The keep/drop decision itself is the device's (moe_dispatch_sharded).
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist


def queue_bases(local_counts: torch.Tensor, group=None):
    """(queue_base [E], batch_counts [E]) from this rank's pre-drop counts [E] (int32): the picks of
    each expert on earlier ranks, and on all ranks."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    c = local_counts.to(torch.int64).contiguous()
    gathered = [torch.empty_like(c) for _ in range(world)]
    dist.all_gather(gathered, c, group=group)
    stack = torch.stack(gathered)                    # [world][E]
    base = stack[:rank].sum(dim=0) if rank > 0 else torch.zeros_like(c)
    return base.to(torch.int32), stack.sum(dim=0)


def aux_loss(local_counts: torch.Tensor, local_psum: torch.Tensor, units_global: int, K: int, alpha: float,
             group=None) -> float:
    """L_aux = α·E·Σ_i f_i·P_i over the whole batch from each rank's pre-drop counts [E] and
    Σ_t p_{t,i} [E] over its units: one all-reduce of the 2E values (float64)."""
    E = local_counts.numel()
    v = torch.cat([local_counts.to(torch.float64), local_psum.to(torch.float64)])
    dist.all_reduce(v, op=dist.ReduceOp.SUM, group=group)
    f = v[:E] / float(units_global * K)
    P = v[E:] / float(units_global)
    return float(alpha * E * torch.sum(f * P).item())

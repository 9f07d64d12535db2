"""Token-sharded data parallelism for the layer: its one exchange step.

A batch split over ranks in token order routes exactly like the whole batch on one GPU once
each rank knows how many assignments every earlier shard sent to each expert, because the
capacity rule keeps the first C arrivals of each expert in token order.  The exchange is one
all_gather of E + 1 int32 per rank (the shard's raw expert counts and its token count); the
dispatch itself, including the prefix over earlier shards, runs in the library's kernel
(moe_dispatch_sharded).  Works on any torch.distributed backend whose all_gather takes
tensors on the counts' device (NCCL for device tensors, gloo for host tensors).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def exchange_counts(counts_raw: torch.Tensor, T_local: int, group=None):
    """All ranks' expert counts and the batch size.

    counts_raw: [E] int32, this shard's assignments per expert before the capacity cut.
    Returns (counts_all [R, E] int32 on counts_raw's device, in rank order; T_global)."""
    E = counts_raw.numel()
    mine = torch.empty(E + 1, dtype=torch.int32, device=counts_raw.device)
    mine[:E].copy_(counts_raw.reshape(-1))
    mine[E:].fill_(int(T_local))
    world = dist.get_world_size(group)
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine, group=group)
    allv = torch.stack(parts)
    T_global = sum(int(v) for v in allv[:, E].cpu().tolist())
    return allv[:, :E].contiguous(), T_global


def sharded_dispatch(topk_idx: torch.Tensor, E: int, capacity_factor: float, group=None,
                     stream=None):
    """Routing of this rank's shard with the whole batch's capacity decisions.

    topk_idx [T, k] int32 on the device (from moe_gate_topk).  Returns a dict with the
    shard's counts_raw, kept, offsets, perm (local token indices), slot_of, counts_all,
    T_global and C."""
    from . import moe_capacity, moe_dispatch, moe_dispatch_sharded

    T, k = topk_idx.shape
    dev = topk_idx.device
    z = lambda n: torch.zeros(n, dtype=torch.int32, device=dev)  # noqa: E731
    counts_raw, kept, offsets = z(E), z(E), z(E + 1)
    perm = z(max(1, T * k))
    slot_of = torch.empty((T, k), dtype=torch.int32, device=dev)
    if T > 0:
        # the shard's own counts (its local drop decisions are replaced below)
        moe_dispatch(topk_idx, E, capacity_factor, counts_raw, kept, offsets, perm, slot_of,
                     stream=stream)
    counts_all, T_global = exchange_counts(counts_raw, T, group)
    rank = dist.get_rank(group)
    moe_dispatch_sharded(topk_idx, E, capacity_factor, T_global, counts_all, rank, counts_raw,
                         kept, offsets, perm, slot_of, stream=stream)
    return dict(counts_raw=counts_raw, kept=kept, offsets=offsets, perm=perm, slot_of=slot_of,
                counts_all=counts_all, T_global=T_global,
                C=moe_capacity(T_global, E, capacity_factor))

"""Batch sharding for runs on several GPUs (one process per GPU).

Batch elements are independent decode problems: each has its own beacon and window
cache, so ranks split the batch and exchange nothing on the data path. Rank r of N
owns the contiguous global batch elements [r * B, (r + 1) * B), where B is the
per-rank batch (weak scaling: per-GPU work stays fixed as N grows).
"""
from __future__ import annotations

from typing import List


def batch_shard(per_rank_batch: int, world: int, rank: int) -> List[int]:
    """Global batch indices owned by ``rank`` of ``world``."""
    if per_rank_batch < 1 or world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad shard request B={per_rank_batch} world={world} rank={rank}")
    return list(range(rank * per_rank_batch, (rank + 1) * per_rank_batch))


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest of every rank's ``value`` (the step time a job is held to)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())

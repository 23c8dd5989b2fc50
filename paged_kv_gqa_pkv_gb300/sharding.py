"""Host-side sharding for multi-GPU runs of independent sequences.

Decode and prefill are independent per sequence, so N ranks each serve their
own shard (weak scaling): rank r draws its batch with seed ``base_seed + r``
and nothing is exchanged on the data path. The only collective is the
max-over-ranks of a timing, taken on the host side of the benchmark.
"""

from __future__ import annotations

import torch


def shard_seed(rank: int, base_seed: int = 0) -> int:
    """Seed of rank `rank`'s shard of the global batch."""
    if rank < 0:
        raise ValueError("rank must be >= 0")
    return base_seed + rank


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over all ranks of the default process group (the
    value itself when torch.distributed is not initialised)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return units_per_rank * world / seconds_max

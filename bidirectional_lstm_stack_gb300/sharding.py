"""Window sharding across ranks (one process per GPU).

Windows are independent (each carries its own zero initial state and the
recurrence never mixes windows), so a batch splits across GPUs with no data
exchange at all: rank r runs windows [start, stop) through its own stack.
The only collective is on timing: the job's step time is the slowest rank's.
"""
from __future__ import annotations


def window_shard(total: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [start, stop) of `total` windows owned by `rank` of `world`.

    Shards differ in size by at most one window; together they cover every
    window exactly once.
    """
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    if total < 0:
        raise ValueError(f"total {total}")
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of `value` over the default process group (itself when
    torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())

"""Host-side request sharding for runs with one process per GPU.

Every part of the hot path is independent per request (sampling, verify) or per position
(accept rate), so a global batch of requests is split into contiguous shards, one per rank,
and each rank runs the whole path on its shard with no collective on the data path.  The only
cross-rank traffic is the timing reduction of the benchmark (the slowest rank defines the step
time).  A budget shared by all ranks' schedulers would need one all-gather of the survival
values; with per-rank budgets (each rank verifies its own shard) there is none.
"""
from __future__ import annotations


def shard_requests(global_B: int, world: int, rank: int) -> tuple[int, int]:
    """(first request, number of requests) of `rank` when `global_B` requests are split into
    `world` contiguous shards whose sizes differ by at most one (lower ranks take the extra)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad rank {rank} of world {world}")
    if global_B < 0:
        raise ValueError("negative batch")
    q, r = divmod(global_B, world)
    start = rank * q + min(rank, r)
    return start, q + (1 if rank < r else 0)


def rank_seed(seed: int, rank: int) -> int:
    """Philox key of a rank's shard: request indices restart at 0 in every call, so each rank
    draws from its own key (seed + rank * 2^32 keeps the low word, moves the high word)."""
    return (int(seed) + (int(rank) << 32)) & (2 ** 64 - 1)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks of the default process group (identity without one)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: list[int] | int, world: int, step_seconds: float) -> float:
    """Units processed by all ranks per second, the step time being the slowest rank's."""
    total = sum(units_per_rank) if isinstance(units_per_rank, list) else units_per_rank * world
    return total / step_seconds

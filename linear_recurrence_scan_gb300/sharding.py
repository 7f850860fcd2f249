"""Row sharding across ranks.

Rows (environments) of a rollout buffer are independent recurrences, so a
batch splits across GPUs by rows with no data exchange: each rank scans its
own contiguous block of rows.  The only collective is the benchmark's
max-over-ranks of the step time.
"""
from __future__ import annotations


def shard_rows(num_envs: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous row block [start, stop) of `rank` out of `world` ranks;
    block sizes differ by at most one row."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world of size {world}")
    if num_envs < 0:
        raise ValueError("num_envs must be >= 0")
    base, extra = divmod(num_envs, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float) -> float:
    """Maximum of a per-rank scalar over the default process group (the
    value itself when no group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())

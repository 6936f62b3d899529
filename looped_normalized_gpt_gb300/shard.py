"""Host logic of multi-GPU runs: one process per GPU, sequences sharded across ranks.

Decode batches and prefill shard by sequence: every rank holds the whole model and the
KV state of its own sequences, so there is no exchange on the data path. Batch-1 decode
does not shard (every norm needs the whole vector): each rank then runs a replica. The
only collective is the timing: ranks meet at a barrier around the timed region and the
slowest rank's time counts.
"""
from __future__ import annotations


def shard(n: int, rank: int, world: int) -> range:
    """The contiguous block of n items (sequences) rank `rank` of `world` owns."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    a = n * rank // world
    b = n * (rank + 1) // world
    return range(a, b)


def slowest(ms: float, group=None) -> float:
    """Max of a per-rank time over all ranks (the time the whole job took)."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64)
    if dist.get_backend(group) == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def job_throughput(units_per_rank: list[int] | int, ms_slowest: float, world: int) -> float:
    """Units all ranks processed per second of the slowest rank's time."""
    total = sum(units_per_rank) if isinstance(units_per_rank, list) else units_per_rank * world
    return total / (ms_slowest / 1e3)

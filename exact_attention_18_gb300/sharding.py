"""Data-parallel layout of the attention hot path across ranks.

Every (b, h) head of the forward and the backward is independent
("fa-triton" §Grid 与并行策略; "T5 讲解" §②), so a job shards the flattened
B*H axis of its [B, H, S, D] tensors into contiguous ranges, one per rank,
and each rank calls the library on its range (a [1, count, S, D] view that
starts `start * S * D` elements into each tensor).  No collective touches
the data; the only cross-rank step is the benchmark's max-over-ranks time.

Sequence (context) sharding splits the keys instead: rank r holds keys
`shard_keys(S, r, world)`, computes every query's partial output and
logsumexp over its keys, and the partials meet in the logsumexp merge
(`fa_merge_lse`; "T5 讲解" §⑥ on merging shards by L).  That exchange is the
one collective such a layout needs; this module only fixes the key ranges.
"""
from __future__ import annotations


def shard_heads(bh: int, rank: int, world: int) -> tuple[int, int]:
    """(start, count) of rank's contiguous share of `bh` heads; the first
    bh % world ranks take one extra head.  Shares are disjoint and cover
    [0, bh) in rank order."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} is not in a world of {world}")
    if bh < 0:
        raise ValueError("negative head count")
    base, extra = divmod(bh, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def shard_keys(S: int, rank: int, world: int, align: int = 128) -> tuple[int, int]:
    """[k0, k1) of rank's share of S keys in contiguous ranges whose starts are
    multiples of `align` (the split-KV shard granularity); later ranks may get
    an empty range when S is small."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} is not in a world of {world}")
    if S < 0 or align <= 0:
        raise ValueError("negative key count or bad alignment")
    per = (S + world - 1) // world
    per = (per + align - 1) // align * align
    k0 = min(S, rank * per)
    return k0, min(S, k0 + per)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the
    job's time is its slowest rank's); `value` itself without one."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job rate: the units all ranks processed over the slowest rank's
    time, per second (units / s)."""
    if max_ms <= 0:
        raise ValueError("time must be positive")
    return world * units_per_rank_step * steps / (max_ms * 1e-3)

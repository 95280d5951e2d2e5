"""Host-side logic of the multi-GPU path (one process per GPU).

Paged attention shards with no exchange: every (sequence, KV head) unit is
independent, so each rank runs the whole hot path on its own GPU over its
own sequences (weak scaling: a fixed batch per GPU), or over a contiguous
share of one batch's sequences (strong scaling).  The only communication is
host-side bookkeeping: a barrier around the timed region and the maximum of
the per-rank step times.  There is no data-path collective.
"""
from __future__ import annotations

from typing import List, Tuple


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s independent batch (rank 0 keeps the base seed)."""
    return int(base_seed) + 7919 * int(rank)


def shard_sequences(lengths: List[int], world: int, rank: int) -> Tuple[int, int]:
    """Contiguous range [lo, hi) of sequences for `rank` so that every rank gets
    about the same number of KV tokens (greedy cut of the length prefix)."""
    if world <= 0 or not (0 <= rank < world):
        raise ValueError("bad world / rank")
    total = sum(int(x) for x in lengths)
    cuts = [0]
    acc = 0
    target_idx = 1
    for i, x in enumerate(lengths):
        acc += int(x)
        while target_idx < world and acc * world >= target_idx * total and len(cuts) <= target_idx:
            cuts.append(i + 1)
            target_idx += 1
    while len(cuts) < world:
        cuts.append(len(lengths))
    cuts.append(len(lengths))
    return cuts[rank], cuts[rank + 1]


def max_over_ranks(values: List[float], group=None) -> List[float]:
    """Element-wise maximum of per-rank timings (torch.distributed all_reduce
    MAX on the host, any backend)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        if dist.get_backend(group) == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return [float(x) for x in t.cpu()]


def aggregate_throughput(work_per_rank: float, world: int, step_ms: float, unit_scale: float) -> float:
    """Whole-job throughput: the work every rank did divided by the slowest
    rank's step time (unit_scale 1e9 for GB/s, 1e12 for TFLOP/s)."""
    return work_per_rank * world / (step_ms * 1e-3) / unit_scale

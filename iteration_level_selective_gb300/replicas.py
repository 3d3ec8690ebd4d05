"""Replicas across GPUs: one independent engine per rank, no data-path collective.

A selectively batched iteration couples requests only through one
engine's scheduler state, so N GPUs serve N independent request streams.
The process group is used only around the timed region: a barrier before
it, then the slowest rank's time (MAX) and the summed work counts (SUM)
after it, so whole-job throughput = total work / slowest time.
"""
from __future__ import annotations

from typing import Sequence, Tuple


def trace_seed(rank: int, generation: int = 0) -> int:
    """Seed of rank `rank`'s synthetic request stream (distinct per rank)."""
    return 1000 * rank + generation


def reduce_timing(seconds: Sequence[float], counts: Sequence[float], device=None) -> Tuple[list, list]:
    """MAX-reduce the timings and SUM-reduce the counts over the default
    process group (identity when it is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(seconds), list(counts)
    t = torch.tensor(list(seconds), dtype=torch.float64, device=device)
    c = torch.tensor(list(counts), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    return t.tolist(), c.tolist()

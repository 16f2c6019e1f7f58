"""Host-side helpers for running the path on several GPUs, one process each.

Attention over a paged KV cache has no exchange step between sequences or KV
heads, so the path shards by rows with no data-path collective: each rank
runs its own batch on its own GPU.  The only collectives are the benchmark's
barrier and the max-over-ranks reduction of the measured time.
"""
from __future__ import annotations

import os
from typing import List, Sequence

import torch
import torch.distributed as dist


def env_rank_world():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def shard_rows(num_rows: int, rank: int, world: int) -> List[int]:
    """Contiguous, balanced split of row indices (rank r gets rows
    [r*n//w, (r+1)*n//w))."""
    lo = rank * num_rows // world
    hi = (rank + 1) * num_rows // world
    return list(range(lo, hi))


def shard_rows_by_work(work: Sequence[int], world: int) -> List[List[int]]:
    """Greedy longest-first assignment of rows to ranks by work (deterministic)."""
    order = sorted(range(len(work)), key=lambda i: (-work[i], i))
    loads = [0] * world
    out: List[List[int]] = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda k: (loads[k], k))
        out[r].append(i)
        loads[r] += work[i]
    return [sorted(x) for x in out]


def init(backend: str):
    if dist.is_available() and not dist.is_initialized() and int(os.environ.get("WORLD_SIZE", "1")) > 1:
        dist.init_process_group(backend=backend)


def barrier():
    if dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    if not dist.is_initialized():
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    if not dist.is_initialized():
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())

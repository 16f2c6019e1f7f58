"""Multi-rank host logic on the CPU (gloo, world size 2).

Rows are independent problems, so several GPUs run disjoint row sets (or
independent replicas) with no collective on the data path; the only
collectives are the benchmark's barrier and max-over-ranks timing.  These
tests run those pieces as two CPU processes.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_attention_prefill_gb300 import dist as padist


def test_shard_rows_covers_each_row_once():
    for n in (0, 1, 7, 256):
        for w in (1, 2, 3, 8):
            got = [r for k in range(w) for r in padist.shard_rows(n, k, w)]
            assert got == list(range(n))


def test_shard_rows_by_work_balances_and_covers():
    work = [17281, 16999, 4320, 11463, 10800, 1302, 7294, 15833]
    parts = padist.shard_rows_by_work(work, 2)
    assert sorted(r for p in parts for r in p) == list(range(len(work)))
    loads = [sum(work[r] for r in p) for p in parts]
    assert max(loads) - min(loads) <= max(work)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    padist.init("gloo")
    try:
        r, w, lr = padist.env_rank_world()
        assert (r, w, lr) == (rank, world, rank)
        padist.barrier()
        # each rank "times" its own shard; the reported time is the max
        t = padist.max_over_ranks(1.5 + rank)
        units = padist.sum_over_ranks(100.0 * (rank + 1))
        rows = padist.shard_rows(10, rank, world)
        q.put((rank, t, units, rows))
    finally:
        dist.destroy_process_group()


def test_two_rank_barrier_and_reductions():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [x[1] for x in res] == [2.5, 2.5]          # max over ranks
    assert [x[2] for x in res] == [300.0, 300.0]      # sum over ranks
    assert res[0][3] + res[1][3] == list(range(10))   # disjoint, complete shards


def test_single_process_helpers_are_identity():
    assert padist.max_over_ranks(3.0) == 3.0
    assert padist.sum_over_ranks(3.0) == 3.0
    padist.barrier()  # no process group: a no-op

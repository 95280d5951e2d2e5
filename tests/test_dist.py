"""Multi-process (gloo, world size 2) checks of the host logic of the N>1 path:
independent batches per rank, max-over-ranks timing, whole-job throughput,
and a token-balanced split of one batch across ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_attention_gb300 import dist as D
from paged_attention_gb300 import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.decode_bf16(mtp=1, shrink=32, seed=D.rank_seed(1002, rank))
        # each rank's own batch differs (independent work, no exchange)
        sig = float(w.q.float().sum())
        ms = [1.0 + rank, 10.0 - rank]
        mx = D.max_over_ranks(ms)
        dist.barrier()
        gathered = [None] * world
        dist.all_gather_object(gathered, sig)
        q.put((rank, mx, gathered,
               D.aggregate_throughput(1e9, world, mx[0], 1e9)))
    finally:
        dist.destroy_process_group()


def test_two_rank_weak_scaling_bookkeeping():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, mx, gathered, thr in res:
        assert mx == [2.0, 10.0]                 # max over ranks, element-wise
        assert gathered[0] != gathered[1]        # independent batches
        assert thr == pytest.approx(2 * 1e9 / 2e-3 / 1e9)


def test_rank_seed_distinct():
    assert D.rank_seed(5, 0) == 5
    assert len({D.rank_seed(5, r) for r in range(8)}) == 8


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_sequences_partition(world):
    g = torch.Generator().manual_seed(3)
    lens = W._log_uniform_ints(64, 128, 32768, g)
    ranges = [D.shard_sequences(lens, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == len(lens)
    for (a, b), (c, d) in zip(ranges, ranges[1:]):
        assert b == c and a <= b
    total = sum(lens)
    for a, b in ranges:
        # every rank is within one sequence of its fair share
        assert abs(sum(lens[a:b]) - total / world) <= max(lens) + 1

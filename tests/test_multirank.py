"""The multi-GPU host logic (replicas with a request partition) on two gloo
ranks on the CPU: disjoint request shares, per-rank batches, the
max-over-ranks time and the whole-job throughput."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_top_kv_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        share = list(replicas.partition_requests(64, world, rank))
        order = replicas.rank_request_order(64, rank).tolist()
        # Rank r "took" 10 + r ms; the job's time is the slowest rank's.
        t = replicas.max_over_ranks(10.0 + rank)
        stats = replicas.sum_over_ranks(torch.tensor([100 + rank, 7], dtype=torch.int64))
        gathered = [None] * world
        dist.all_gather_object(gathered, share)
        q.put((rank, share, order, t, stats.tolist(), gathered))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, share, order, t, stats, gathered = q.get(timeout=120)
        res[rank] = (share, order, t, stats, gathered)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # Disjoint shares that cover all requests, seen identically by both ranks.
    s0, s1 = res[0][0], res[1][0]
    assert sorted(s0 + s1) == list(range(64)) and not set(s0) & set(s1)
    assert res[0][4] == res[1][4] == [s0, s1]
    # Weak scaling: rank 0 keeps the order, rank 1 serves a permuted batch.
    assert res[0][1] == list(range(64))
    assert sorted(res[1][1]) == list(range(64)) and res[1][1] != list(range(64))
    # Max over ranks and summed counters agree on both ranks.
    assert res[0][2] == res[1][2] == 11.0
    assert res[0][3] == res[1][3] == [201, 14]
    assert replicas.whole_job_throughput(13, world, 11.0) == pytest.approx(2 * 13 / 0.011)


@pytest.mark.parametrize("n,world", [(64, 1), (64, 3), (5, 8), (0, 2), (130, 7)])
def test_partition_is_balanced(n, world):
    shares = [replicas.partition_requests(n, world, r) for r in range(world)]
    flat = [i for s in shares for i in s]
    assert flat == list(range(n))
    sizes = [len(s) for s in shares]
    assert max(sizes) - min(sizes) <= 1


def test_single_process_is_identity():
    assert replicas.max_over_ranks(3.5) == 3.5
    c = torch.tensor([1, 2])
    assert replicas.sum_over_ranks(c).tolist() == [1, 2]
    assert np.array_equal(replicas.rank_request_order(8, 0), np.arange(8))

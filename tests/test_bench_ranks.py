"""The multi-rank form of bench.py on CPU: two gloo ranks (one process each, as torchrun
launches them) draw different blocks of the same workload with the same weights, take
the slowest rank's time and report the whole-job throughput."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = bench.rank_workload("tiny", None, 3, rank)
        # every rank's logits digest and weights digest, gathered on all ranks
        dig = torch.tensor([float(np.abs(wl.logits).sum()),
                            float(sum(np.abs(v).sum() for v in wl.weights.values()))],
                           dtype=torch.float64)
        allg = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(allg, dig)
        local_s = 0.5 + rank  # rank 1 is the slower one
        slowest = bench.max_over_ranks(local_s, "cpu")
        value = bench.job_throughput(wl.batch, 10, world, slowest)
        q.put((rank, wl.batch, [t.tolist() for t in allg], slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, batch, allg, slowest, value in res:
        assert batch == 3
        (l0, w0), (l1, w1) = allg
        assert l0 != l1, "ranks must process different blocks"
        assert w0 == w1, "ranks must share one model"
        assert slowest == 1.5  # the max over ranks, seen by every rank
        assert value == pytest.approx(3 * 10 * world / 1.5)


def test_single_rank_helpers_without_a_process_group():
    assert bench.max_over_ranks(0.25, "cpu") == 0.25
    assert bench.job_throughput(256, 200, 1, 0.25) == pytest.approx(204800.0)
    a = bench.rank_workload("tiny", None, 2, 0)
    b = bench.rank_workload("tiny", None, 2, 0)
    assert np.array_equal(a.logits, b.logits)

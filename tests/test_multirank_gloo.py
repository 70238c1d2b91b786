"""The benchmark's multi-rank host logic on CPU with world_size 2 (gloo):
max over ranks of the per-rank timings, weak-scaling rate, and that a
collective-free replica step gives each rank its own, identical result."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], world)
        rate = bench.whole_job_rate(1000, world, max(got[0], 1e-9))
        # a replica step: the oracle's plan of the same batch on every rank,
        # no data-path collective; the ranks compare totals afterwards
        import numpy as np
        import oracle
        from deepseek_v4_compressed_c2_gb300 import workloads as W
        cfg = W.cfg2_ratio2_small()
        total = oracle.plan(2, cfg["ext"], cfg["page_table"], cfg["page_bits"])["total"]
        t = torch.tensor([total], dtype=torch.int64)
        dist.all_reduce(t, op=dist.ReduceOp.MIN)
        q.put((rank, got, rate, total, int(t.item())))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate, total, tmin in res:
        assert got == [2.0, 10.0, 3.5]                 # element-wise max of both ranks
        assert rate == pytest.approx(1000 * world / (2.0 / 1e3))
        assert total == tmin == 1809


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.whole_job_rate(10, 1, 5.0) == pytest.approx(2000.0)

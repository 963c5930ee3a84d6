"""The benchmark's multi-rank aggregation (max over ranks of the timed
region, weak-scaling whole-job throughput) on a world-size-2 gloo group on
CPU: the path has no data-path collective, only this timing reduction."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [120.0, 150.0][rank]          # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed)
    v = bench.weak_scaling_throughput(16384, 10, world, m)
    out[rank] = (m, v)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        m, v = out[r]
        assert m == 150.0
        assert v == pytest.approx(2 * 16384 * 10 / 0.150)


def test_single_process_passthrough():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.weak_scaling_throughput(100, 2, 1, 1000.0) == pytest.approx(200.0)

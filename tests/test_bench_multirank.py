"""The benchmark's multi-rank path on CPU: two gloo ranks take the maximum
of their timings and report whole-job throughput (independent replicas, no
data-path collective)."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [12.5, 14.0][rank]
    got = bench.reduce_max(ms, dist, "cpu")
    thr = bench.job_throughput(world, 1000.0, got)
    q.put((rank, got, thr))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, thr in results:
        assert got == 14.0
        assert thr == pytest.approx(2 * 1000.0 / 0.014)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, None, "cpu") == 3.5
    assert bench.job_throughput(1, 10.0, 2.0) == pytest.approx(5000.0)

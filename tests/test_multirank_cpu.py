"""The benchmark's multi-rank path on the CPU: two gloo ranks, each with its
own elapsed time and work, reduce to the slowest rank's time and the summed
work (weak scaling: every rank runs its own copy of the workload; the
operator's data path has no collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        elapsed = [0.25, 0.5][rank]
        units = [100.0, 300.0][rank]
        bench.barrier(world)
        t, u = bench.reduce_timing(elapsed, units, world, device=torch.device("cpu"))
        q.put((rank, t, u))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_time_and_total_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, u in got:
        assert t == pytest.approx(0.5) and u == pytest.approx(400.0)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_timing(1.5, 7.0, 1) == (1.5, 7.0)


def _regions_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cpu = torch.device("cpu")
        # the ranks' first regions differ; every rank must time the same count
        n = bench.region_count([0.004, 0.01, 0.002][rank], world, cpu)
        elapsed = [[0.01, 0.02, 0.03], [0.03, 0.01, 0.02], [0.02, 0.02, 0.01]][rank]
        reg, units = bench.reduce_regions(elapsed, [10.0, 20.0, 30.0][rank], world, cpu)
        q.put((rank, n, reg, units))
    finally:
        dist.destroy_process_group()


def test_three_gloo_ranks_agree_on_regions_and_reduce_each():
    """Timed regions under torchrun: the count comes from the slowest rank's
    first region (at least 5, about 100 ms in all), each region's time is the
    slowest rank's, and the work units are summed."""
    world = 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_regions_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, n, reg, units in got:
        assert n == 10  # 100 ms over the slowest first region (10 ms)
        assert reg == pytest.approx([0.03, 0.02, 0.03]) and units == pytest.approx(60.0)


def test_region_count_bounds():
    import bench
    assert bench.region_count(1.0, 1) == 5          # long regions: at least 5
    assert bench.region_count(1e-6, 1) == 200       # tiny regions: capped
    assert bench.region_count(0.0039, 1) == 26      # the default run's 3.9 ms regions

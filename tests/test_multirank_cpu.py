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

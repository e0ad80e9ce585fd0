"""The data-parallel token split on the CPU: rope_partial_token_shard's
ranges and runs (host logic of the C ABI, no GPU), and gloo ranks (world
sizes 2 and 3) that each rotate only their own tokens with their own cos/sin
rows, whose pieces put together are bit-identical to one rank rotating the
whole workload.  The rotation on each rank is the CPU oracle, so this checks
the split, the run views and the per-rank cos/sin rows; the GPU tests check
the kernels."""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from place_partial_rope_gb300 import binding, build, shard, synth


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.load_library()


@pytest.mark.parametrize("B,S", [(1, 1), (1, 7), (3, 5), (2, 7), (4, 8192), (5, 3), (7, 1),
                                 (0, 4), (3, 0)])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_shares_tile_the_tokens(B, S, world):
    T = B * S
    prev = 0
    for rank in range(world):
        sh = shard.token_share(B, S, rank, world)
        assert sh.t0 == prev and sh.t1 >= sh.t0
        assert sh.tokens in (T // world, T // world + 1)
        assert sh.tokens == T // world + (1 if rank < T % world else 0)
        prev = sh.t1
        t = sh.t0
        assert len(sh.runs) <= 3 and (len(sh.runs) > 0) == (sh.tokens > 0)
        for run in sh.runs:
            # each run is one contiguous block of a BSND tensor, in token order
            assert run.b0 * S + run.s0 == t and run.tokens > 0
            assert run.nb == 1 or (run.s0 == 0 and run.ns == S)
            assert 0 <= run.s0 and run.s0 + run.ns <= S and run.b0 + run.nb <= B
            t += run.tokens
        assert t == sh.t1
    assert prev == T


def test_rejected_shares(lib):
    import ctypes
    t0, t1, n = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    runs = (binding.RopeTokenRun * 3)()
    args = (ctypes.byref(t0), ctypes.byref(t1), runs, ctypes.byref(n))
    assert lib.rope_partial_token_shard(2, 3, 2, 2, *args) == binding.ROPE_ERR_INVALID
    assert lib.rope_partial_token_shard(2, 3, -1, 2, *args) == binding.ROPE_ERR_INVALID
    assert lib.rope_partial_token_shard(2, 3, 0, 0, *args) == binding.ROPE_ERR_INVALID
    assert lib.rope_partial_token_shard(-1, 3, 0, 1, *args) == binding.ROPE_ERR_INVALID
    assert lib.rope_partial_token_shard(2**40, 2**40, 0, 1, *args) == binding.ROPE_ERR_INVALID
    assert lib.rope_partial_token_shard(2, 3, 0, 1, None, ctypes.byref(t1), runs,
                                        ctypes.byref(n)) == binding.ROPE_ERR_NULLPTR


# small workloads with the named workloads' position rules and cos/sin forms
_L = synth.WORKLOADS["large_unaligned"]
SMALL = [
    dataclasses.replace(_L, name="per_batch_offsets", shape=(3, 5, 2, 16), start=2, end=12,
                        r_shape=(3, 5, 1, 10)),
    dataclasses.replace(synth.WORKLOADS["gqa"], name="shared_positions", shape=(2, 7, 3, 8),
                        start=0, end=8, r_shape=(1, 7, 1, 8)),
    dataclasses.replace(synth.WORKLOADS["mla_decode_q"], name="per_token", shape=(7, 1, 2, 12),
                        start=0, end=6, r_shape=(7, 1, 1, 6)),
    dataclasses.replace(_L, name="per_batch_offsets_bf16", dtype="bf16", shape=(2, 7, 2, 10),
                        start=3, end=9, r_shape=(2, 7, 1, 6)),
]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_pieces(w, rank, world):
    """This rank's rotated tokens (forward and backward), from its share of
    the global inputs and its runs' cos/sin rows, through the oracle."""
    import oracle
    x, r1, r2, g = synth.workload_inputs(w)
    g = g if g is not None else synth.normal(w.shape, w.dtype, w.seed + 500)
    B, S, N, D = w.shape
    sh = shard.token_share(B, S, rank, world)
    xs = x.reshape(B * S, N, D)[sh.t0:sh.t1].copy()
    gs = g.reshape(B * S, N, D)[sh.t0:sh.t1].copy()
    # the per-rank inputs bench.py builds: its cos/sin rows, from positions
    ri = shard.rank_inputs(w, rank, world, weak=False)
    for run, (c, s) in zip(sh.runs, ri.tables):
        want_c, want_s = shard.run_rows(r1, run), shard.run_rows(r2, run)
        assert c.shape == want_c.shape and np.array_equal(c, want_c)
        assert np.array_equal(s, want_s)
        for buf, fn in ((xs, oracle.fwd), (gs, oracle.bwd)):
            blk = shard.run_block(buf, sh, run)
            blk[...] = fn(np.ascontiguousarray(blk), c, s, w.dtype, w.start, w.end)
    return sh.t0, sh.t1, xs, gs


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for k, w in enumerate(SMALL):
            piece = _rank_pieces(w, rank, world)
            got = [None] * world
            dist.all_gather_object(got, piece)
            if rank == 0:
                q.put((k, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_rotate_their_tokens(world):
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=300) for _ in SMALL)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for k, w in enumerate(SMALL):
        B, S, N, D = w.shape
        x, r1, r2, g = synth.workload_inputs(w)
        g = g if g is not None else synth.normal(w.shape, w.dtype, w.seed + 500)
        pieces = sorted(results[k], key=lambda p: p[0])
        assert pieces[0][0] == 0 and pieces[-1][1] == B * S
        assert all(a[1] == b[0] for a, b in zip(pieces, pieces[1:]))  # the ranges tile [0, B*S)
        view = np.uint32 if w.dtype == "fp32" else np.uint16
        got_x = np.concatenate([p[2] for p in pieces]).reshape(w.shape)
        got_g = np.concatenate([p[3] for p in pieces]).reshape(w.shape)
        assert np.array_equal(got_x.view(view), oracle.fwd(x, r1, r2, w.dtype, w.start, w.end).view(view)), w.name
        assert np.array_equal(got_g.view(view), oracle.bwd(g, r1, r2, w.dtype, w.start, w.end).view(view)), w.name


@pytest.mark.parametrize("name", ["tiny", "small_model"])
def test_one_rank_holds_the_named_workload(name):
    """With one rank the rank's inputs are the named workload's, value for value."""
    w = synth.WORKLOADS[name]
    x, r1, r2, g = synth.workload_inputs(w)
    ri = shard.rank_inputs(w, 0, 1)
    assert ri.workload == w and len(ri.share.runs) == 1
    assert np.array_equal(ri.x.reshape(w.shape).view(np.uint8), x.view(np.uint8))
    assert (ri.g is None) == (g is None) and (g is None or np.array_equal(ri.g.reshape(w.shape), g))
    assert np.array_equal(ri.tables[0][0], r1) and np.array_equal(ri.tables[0][1], r2)
    assert ri.algorithmic_bytes() == w.algorithmic_bytes()


def test_weak_scaling_gives_each_rank_the_named_workload_size():
    w = synth.WORKLOADS["large_unaligned"]
    for world in (2, 4, 8):
        wg = shard.weak_workload(w, world)
        assert wg.shape == (4 * world, 8192, 32, 128) and wg.r_shape == (4 * world, 8192, 1, 64)
        for rank in range(world):
            sh = shard.token_share(*wg.shape[:2], rank, world)
            assert sh.tokens == 4 * 8192 and len(sh.runs) == 1 and sh.runs[0].nb == 4
    g = shard.weak_workload(synth.WORKLOADS["gqa"], 4)
    assert g.shape == (128, 2048, 16, 128) and g.r_shape == (1, 2048, 1, 64)


def test_bench_rank_calls_cover_each_run_in_order():
    """bench.py's step on one rank: every direction over every run of the
    rank's share, forward first, each on the run's block of the rank's
    buffer and the run's own cos/sin rows (a fake binding records them)."""
    import torch

    import bench

    class Fake:
        calls = []

        @staticmethod
        def _rec(name):
            def prep(buf, c, s, start, end):
                Fake.calls.append((name, tuple(buf.shape), buf.data_ptr(), tuple(c.shape), start, end))
                return lambda: None
            return prep

    Fake.prepare_fwd, Fake.prepare_bwd = Fake._rec("fwd"), Fake._rec("bwd")
    Fake.prepare_fwd_host, Fake.prepare_bwd_host = Fake._rec("fwd_host"), Fake._rec("bwd_host")
    w = SMALL[3]  # (2, 7, 2, 10) [3, 9), per-batch cos/sin rows, forward and backward
    for world in (1, 3):
        for rank in range(world):
            ri = shard.rank_inputs(w, rank, world, weak=False)
            x, g = torch.from_numpy(ri.x.view(np.int16)), torch.from_numpy(ri.g.view(np.int16))
            tabs = [(torch.from_numpy(c.view(np.int16)), torch.from_numpy(s.view(np.int16)))
                    for c, s in ri.tables]
            for host in (False, True):
                Fake.calls = []
                calls = bench.rank_calls(Fake, shard, ri, {"fwd": x, "bwd": g}, tabs, w, host=host)
                n = len(ri.share.runs)
                assert len(calls) == 2 * n
                assert [c[0] for c in Fake.calls] == (["fwd_host"] * n + ["bwd_host"] * n if host
                                                      else ["fwd"] * n + ["bwd"] * n)
                for k, run in enumerate(ri.share.runs):
                    for rec, buf in ((Fake.calls[k], x), (Fake.calls[n + k], g)):
                        _, shape, ptr, cshape, st, en = rec
                        assert shape == (run.nb, run.ns, 2, 10) and (st, en) == (3, 9)
                        assert ptr == buf.data_ptr() + ri.share.offset(run) * 2 * 10 * 2
                        assert cshape == (run.nb, run.ns, 1, 6)

"""The data-parallel token split on the GPU: each rank's share of a workload
(its runs, through the same per-run calls bench.py makes) is rotated on the
one GPU, rank after rank (no rank waits on another), and the rotated tokens
put together equal the oracle on the whole workload, bit for bit.  Shares
that start or end inside a batch (strong scaling) and whole-batch shares
(weak scaling) are both covered."""
import dataclasses

import numpy as np
import pytest
import torch

import bench
import oracle
from gpu_util import DEV
from place_partial_rope_gb300 import binding, shard, synth

pytestmark = pytest.mark.gpu

_L = synth.WORKLOADS["large_unaligned"]
CASES = [
    # per-batch position offsets, the large shape's slice, a few tokens
    dataclasses.replace(_L, name="per_batch", shape=(3, 37, 4, 128), r_shape=(3, 37, 1, 64)),
    # one shared table (gqa-like), fp16
    dataclasses.replace(synth.WORKLOADS["gqa"], name="shared", shape=(2, 45, 8, 128),
                        r_shape=(1, 45, 1, 64)),
    # one row per token (MLA-decode-like), bf16, forward only
    dataclasses.replace(synth.WORKLOADS["mla_decode_q"], name="per_token", shape=(67, 1, 16, 192),
                        r_shape=(67, 1, 1, 64)),
]


@pytest.mark.parametrize("world", [2, 3, 4])
@pytest.mark.parametrize("k", range(len(CASES)))
@pytest.mark.parametrize("weak", [False, True])
def test_ranks_put_together_match_the_oracle(k, world, weak):
    w = CASES[k]
    wg = shard.weak_workload(w, world) if weak else w
    B, S, N, D = wg.shape
    view = np.uint32 if w.dtype == "fp32" else np.uint16
    got = {"fwd": [], "bwd": []}
    for rank in range(world):
        ri = shard.rank_inputs(w, rank, world, weak=weak)
        xd = synth.to_torch(ri.x, w.dtype).to(DEV)
        gd = synth.to_torch(ri.g, w.dtype).to(DEV) if ri.g is not None else None
        tabs = [(synth.to_torch(c, w.dtype).to(DEV), synth.to_torch(s, w.dtype).to(DEV))
                for c, s in ri.tables]
        for call in bench.rank_calls(binding, shard, ri, {"fwd": xd, "bwd": gd}, tabs, w):
            call()
        torch.cuda.synchronize()
        # the oracle on the same rank inputs, whole share at once per run
        for d, buf, host in (("fwd", xd, ri.x), ("bwd", gd, ri.g)):
            if host is None:
                continue
            want = host.copy()
            fn = oracle.fwd if d == "fwd" else oracle.bwd
            for run, (c, s) in zip(ri.share.runs, ri.tables):
                blk = shard.run_block(want, ri.share, run)
                blk[...] = fn(np.ascontiguousarray(blk), c, s, w.dtype, w.start, w.end)
            got[d].append((ri.share.t0, synth.from_torch(buf), want))
    # the ranks tile the tokens, and every rank's rows match
    for d, pieces in got.items():
        if not pieces:
            continue
        pieces.sort(key=lambda p: p[0])
        assert sum(p[1].shape[0] for p in pieces) == B * S
        for t0, g, want in pieces:
            assert np.array_equal(g.view(view), want.view(view)), (w.name, world, weak, d, t0)


def test_one_rank_share_is_the_named_workload_on_the_gpu():
    """With one rank the calls rotate the named workload's inputs exactly as
    a single call on the whole tensor does."""
    w = CASES[0]
    ri = shard.rank_inputs(w, 0, 1)
    xd = synth.to_torch(ri.x, w.dtype).to(DEV)
    gd = synth.to_torch(ri.g, w.dtype).to(DEV)
    tabs = [(synth.to_torch(c, w.dtype).to(DEV), synth.to_torch(s, w.dtype).to(DEV))
            for c, s in ri.tables]
    for call in bench.rank_calls(binding, shard, ri, {"fwd": xd, "bwd": gd}, tabs, w):
        call()
    x, r1, r2, g = synth.workload_inputs(w)
    xs, gs = synth.to_torch(x, w.dtype).to(DEV), synth.to_torch(g, w.dtype).to(DEV)
    c, s = synth.to_torch(r1, w.dtype).to(DEV), synth.to_torch(r2, w.dtype).to(DEV)
    binding.rope_partial_inplace_fwd(xs, c, s, w.start, w.end)
    binding.rope_partial_inplace_bwd(gs, c, s, w.start, w.end)
    torch.cuda.synchronize()
    assert torch.equal(xd.view(torch.int32), xs.reshape(xd.shape).view(torch.int32))
    assert torch.equal(gd.view(torch.int32), gs.reshape(gd.shape).view(torch.int32))

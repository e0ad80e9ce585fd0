"""Launch-level behaviour on the GPU: the calls are captured into CUDA
graphs and replayed, and calls on separate streams run concurrently, with
results equal to the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_same, to_dev
from place_partial_rope_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def test_calls_captured_in_a_cuda_graph():
    """Forward and backward captured once, replayed three times: the result
    is three forwards / backwards in a row."""
    dtype, shape, st, en = "fp16", (4, 64, 8, 128), 0, 64
    x, r1, r2, g = synth.case(shape, st, en, dtype, "BS1D", seed=61, table="rope")
    xd, gd = to_dev(x, dtype), to_dev(g, dtype)
    c, s = to_dev(r1, dtype), to_dev(r2, dtype)
    # first calls outside capture fill the library's device-attribute caches
    binding.prepare_fwd(xd.clone(), c, s, st, en)()
    binding.prepare_bwd(gd.clone(), c, s, st, en)()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd = binding.prepare_fwd(xd, c, s, st, en)
        bwd = binding.prepare_bwd(gd, c, s, st, en)
        fwd()
        bwd()
    # capture records the launches without running them
    assert_same(synth.from_torch(xd), x, dtype, "capture did not run")
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    want_x, want_g = x, g
    for _ in range(3):
        want_x = oracle.fwd(want_x, r1, r2, dtype, st, en)
        want_g = oracle.bwd(want_g, r1, r2, dtype, st, en)
    assert_same(synth.from_torch(xd), want_x, dtype, "graph fwd x3")
    assert_same(synth.from_torch(gd), want_g, dtype, "graph bwd x3")


def test_concurrent_streams():
    """Eight independent tensors rotated on four streams at once."""
    dtype, shape, st, en = "bf16", (8, 256, 8, 64), 0, 64
    streams = [torch.cuda.Stream() for _ in range(4)]
    cases = [synth.case(shape, st, en, dtype, "BS1D", seed=70 + i) for i in range(8)]
    devs = [(to_dev(x, dtype), to_dev(r1, dtype), to_dev(r2, dtype)) for x, r1, r2, _ in cases]
    torch.cuda.synchronize()
    for i, (xd, c, s) in enumerate(devs):
        with torch.cuda.stream(streams[i % 4]):
            binding.rope_partial_inplace_fwd(xd, c, s, st, en)
    torch.cuda.synchronize()
    for (x, r1, r2, _), (xd, _, _) in zip(cases, devs):
        assert_same(synth.from_torch(xd), oracle.fwd(x, r1, r2, dtype, st, en), dtype, "stream")

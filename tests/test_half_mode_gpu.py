"""GPU parity of the half-split rotary mode (pairs (i, i + L/2)) against the
CPU oracle, bit for bit, including every byte outside the slice.  The sweep
covers both half-split kernels: rows of 2..32 accesses (a power of two),
where the partner access comes from another lane, and the rest, where one
thread holds both halves."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, assert_same, to_dev
from place_partial_rope_gb300 import binding, synth, torch_op

pytestmark = pytest.mark.gpu


def run_half(direction, x, r1, r2, dtype, start, end):
    xd = to_dev(x, dtype)
    fn = binding.rope_partial_inplace_fwd_mode if direction == "fwd" else binding.rope_partial_inplace_bwd_mode
    fn(xd, to_dev(r1, dtype), to_dev(r2, dtype), start, end, "half")
    torch.cuda.synchronize()
    return synth.from_torch(xd)


def oracle_half(direction, x, r1, r2, dtype, start, end):
    fn = oracle.fwd if direction == "fwd" else oracle.bwd
    return fn(x, r1, r2, dtype, start, end, oracle.GATHER_CHAIN, "half")


SWEEP = [
    ((2, 5, 3, 64), 0, 64, "BS1D"),
    ((2, 5, 3, 128), 0, 64, "1S1D"),       # gqa-like: 16-byte chunks per half
    ((2, 5, 3, 64), 8, 40, "B11D"),
    ((2, 5, 3, 64), 2, 58, "BSND"),        # halves of 28 lanes, cos/sin per head
    ((2, 5, 3, 64), 3, 61, "BS1D"),        # odd start
    ((2, 5, 7, 48), 1, 3, "B1ND"),         # L = 2: one pair per row
    ((1, 1, 1, 2), 0, 2, "111D"),          # D = 2
    ((1, 7, 5, 1024), 0, 1024, "1S1D"),    # the largest head dim
    ((2, 3, 13, 24), 6, 22, "1SND"),       # ragged heads
    ((4, 9, 1, 10), 0, 10, "BS1D"),        # N = 1, 5-lane halves
    ((3, 1, 128, 192), 0, 64, "B11D"),     # MLA-like rows
    # rows of 2..32 accesses (a power of two): the partner access comes from
    # another lane of the warp
    ((2, 5, 6, 64), 0, 64, "BSND"),        # cos/sin per head, idle head slots
    ((3, 7, 5, 128), 0, 128, "1S1D"),      # fp32: 32 accesses per row
    ((1, 3, 3, 8), 0, 8, "BS1D"),          # 2 accesses per row
    ((1, 1, 3, 64), 0, 64, "BS1D"),        # 16 work items: a partial warp
    ((1, 3, 5, 32), 0, 32, "B1ND"),        # partial warps, cos/sin per head
    ((2, 3, 4, 40), 4, 36, "BS1D"),        # 16-bit: 8-byte accesses
]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("k", range(len(SWEEP)))
def test_half_sweep(dtype, k):
    shape, st, en, form = SWEEP[k]
    x, r1, r2, g = synth.case(shape, st, en, dtype, form, seed=300 + k)
    for direction, inp in (("fwd", x), ("bwd", g)):
        got = run_half(direction, inp, r1, r2, dtype, st, en)
        assert_same(got, oracle_half(direction, inp, r1, r2, dtype, st, en), dtype,
                    f"half {shape} [{st},{en}) {form} {direction}")


@pytest.mark.parametrize("name,span", [("gqa", None), ("large_unaligned", None),
                                       ("large_unaligned", (0, 96))])
def test_half_named_shapes_full_size(name, span):
    """The gqa and large fp32 shapes in half-split mode with a half-layout
    cos/sin table, forward and backward, every element; the large shape also
    at [0, 96), whose 12 accesses per half run both halves in one thread
    (the benchmark's half-split cases)."""
    w = synth.WORKLOADS[name]
    st, en = span if span else (w.start, w.end)
    x = synth.normal(w.shape, w.dtype, w.seed)
    g = synth.normal(w.shape, w.dtype, w.seed + 500)
    r1, r2 = synth.rope_table(synth.positions(w), en - st, w.dtype, layout="half")
    for direction, inp in (("fwd", x), ("bwd", g)):
        got = run_half(direction, inp, r1, r2, w.dtype, st, en)
        assert_same(got, oracle_half(direction, inp, r1, r2, w.dtype, st, en), w.dtype,
                    f"half {name} [{st},{en}) {direction}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("elem_offset", [0, 1, 2])
def test_half_guard_bands(dtype, elem_offset):
    shape, st, en = (3, 11, 5, 40), 4, 36
    x, r1, r2, _ = synth.case(shape, st, en, dtype, "BS1D", seed=17)
    e = synth.ELEM_BYTES[dtype]
    guard = 4096 // e
    n = x.size
    canary = np.full(guard * 2 + elem_offset + n, 0x5A5A5A5A if e == 4 else 0x5A5A,
                     dtype=np.uint32 if e == 4 else np.uint16)
    canary = canary.view(np.float32) if dtype == "fp32" else canary
    buf = to_dev(canary, dtype)
    lo = guard + elem_offset
    view = buf[lo:lo + n].view(shape)
    view.copy_(synth.to_torch(x, dtype).to(DEV))
    binding.rope_partial_inplace_fwd_mode(view, to_dev(r1, dtype), to_dev(r2, dtype), st, en, "half")
    torch.cuda.synchronize()
    host = synth.from_torch(buf)
    assert_same(host[lo:lo + n].reshape(shape), oracle_half("fwd", x, r1, r2, dtype, st, en), dtype,
                "half guard")
    assert np.array_equal(host[:lo], canary[:lo]) and np.array_equal(host[lo + n:], canary[lo + n:])


def test_half_through_the_torch_op_with_autograd():
    dtype = "fp16"
    shape, st, en = (2, 32, 8, 128), 0, 64
    x, r1, r2, g = synth.case(shape, st, en, dtype, "BS1D", seed=23)
    xd = to_dev(x, dtype).requires_grad_(True)
    w = to_dev(g, dtype)
    y = xd * 1.0
    torch_op.inplace_partial_rotary_mul(y, to_dev(r1, dtype), to_dev(r2, dtype), rotary_mode="half",
                                        partial_slice=[st, en])
    (y * w).sum().backward()
    torch.cuda.synchronize()
    assert_same(synth.from_torch(y.detach()), oracle_half("fwd", x, r1, r2, dtype, st, en), dtype, "y")
    assert_same(synth.from_torch(xd.grad), oracle_half("bwd", g, r1, r2, dtype, st, en), dtype, "x.grad")

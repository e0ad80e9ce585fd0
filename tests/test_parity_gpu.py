"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: bit-exact for bf16, fp16 and fp32 (both sides compute each product and
sum as one fp32 rounding and round once to the storage type), including
every byte outside [start, end).  NaN matches NaN.  The five named workloads
and the odd-start cases the benchmark times run at full size and are
compared on every element; a sweep of small seeded cases covers every dtype,
broadcast form, aligned / unaligned / odd slice, ragged head counts and the
degenerate shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, assert_same, run_cuda, run_oracle, to_dev
from place_partial_rope_gb300 import binding, synth

pytestmark = pytest.mark.gpu

NAMED = [(name, d) for name, w in synth.WORKLOADS.items() for d in w.directions]


@pytest.mark.parametrize("name,direction", NAMED)
def test_named_workload_full_size(name, direction):
    w = synth.WORKLOADS[name]
    x, r1, r2, g = synth.workload_inputs(w)
    inp = x if direction == "fwd" else g
    got = run_cuda(direction, inp, r1, r2, w.dtype, w.start, w.end)
    want = run_oracle(direction, inp, r1, r2, w.dtype, w.start, w.end)
    assert_same(got, want, w.dtype, f"{name} {direction}")


SWEEP = [
    # shape, start, end, broadcast form
    ((2, 5, 3, 64), 0, 64, "BS1D"),
    ((2, 5, 3, 64), 0, 32, "1S1D"),
    ((2, 5, 3, 64), 8, 40, "B11D"),
    ((2, 5, 3, 64), 2, 58, "111D"),       # 4-byte (16-bit) / 8-byte (fp32) slice offset
    ((2, 5, 3, 64), 34, 62, "BSND"),      # cos/sin per head
    ((2, 5, 3, 64), 3, 61, "BS1D"),       # odd start
    ((2, 5, 7, 48), 1, 3, "B1ND"),        # one pair per row, odd start
    ((1, 1, 1, 2), 0, 2, "111D"),         # D = 2
    ((3, 1, 1, 6), 4, 6, "B11D"),         # 12-byte rows
    ((1, 7, 5, 1024), 0, 1024, "1S1D"),   # the largest head dim, full slice
    ((1, 3, 2, 1024), 2, 1024, "BSND"),   # L = 1022
    ((2, 3, 13, 24), 6, 22, "1SND"),      # ragged heads (13 = 4 * 4 - 3)
    ((4, 9, 1, 10), 0, 10, "BS1D"),       # N = 1, 20-byte rows
    ((5, 2, 33, 30), 10, 20, "11ND"),     # N = 33
    ((1, 300, 3, 128), 0, 64, "1S1D"),    # several blocks of work
    ((3, 1, 128, 192), 0, 64, "B11D"),    # MLA-like rows of 192
]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("k", range(len(SWEEP)))
def test_sweep(dtype, k):
    shape, st, en, form = SWEEP[k]
    x, r1, r2, g = synth.case(shape, st, en, dtype, form, seed=100 + k)
    for direction, inp in (("fwd", x), ("bwd", g)):
        got = run_cuda(direction, inp, r1, r2, dtype, st, en)
        want = run_oracle(direction, inp, r1, r2, dtype, st, en)
        assert_same(got, want, dtype, f"{shape} [{st},{en}) {form} {direction}")


ODD_STARTS = [
    # shape, start, end, broadcast form, x's element offset in its buffer.
    # An odd start at element 1 of an aligned 16- or 8-byte vector of x runs
    # a lane per vector (path 4; fp32 rows take any odd start at 8 bytes),
    # any other odd start the element path (path 2); odd_path() below states
    # the rule.  Cases: the last lane storing part
    # of its vector, the slice ending one element before the row's end, idle
    # head slots, cos/sin per head, one pair per row, rows whose lanes
    # straddle two warps, and x aligned to 16, 8 or 4 bytes only.
    ((2, 5, 3, 64), 1, 63, "BS1D", 0),       # 31 pairs; ends at D - 1
    ((2, 5, 3, 64), 3, 35, "B11D", 0),       # 16 pairs from element 3
    ((2, 5, 6, 64), 5, 17, "1S1D", 0),       # 6 pairs from element 5; 6 heads
    ((2, 4, 5, 40), 7, 39, "BSND", 0),       # from element 7; cos/sin per head
    ((1, 3, 9, 8), 1, 7, "1SND", 0),         # 3 pairs, cos/sin per head
    ((3, 2, 4, 4), 1, 3, "B1ND", 0),         # one pair per row, ends at D - 1
    ((1, 7, 2, 1024), 1, 1023, "1S1D", 0),   # the longest odd slice: rows span warps
    ((2, 3, 16, 128), 33, 97, "BS1D", 0),    # gqa-like rows, 32 pairs
    ((2, 3, 13, 66), 1, 65, "BS1D", 0),      # 13 heads (idle slots), 132-byte rows
    ((1, 5, 6, 20), 3, 19, "BSND", 0),       # 8 pairs, cos/sin per head
    ((3, 7, 5, 48), 1, 41, "BS1D", 0),       # 5 or 10 lanes per row: rows straddle warps
    ((2, 3, 7, 64), 17, 59, "BS1D", 0),      # 21 pairs: 6 or 11 lanes per row
    ((2, 9, 7, 48), 3, 45, "11ND", 0),       # cos/sin per head
    ((2, 9, 7, 40), 3, 37, "B11D", 2),       # x 4-byte (16-bit) / 8-byte (fp32) aligned
    ((2, 9, 7, 40), 5, 35, "1S1D", 4),       # x 8-byte / 16-byte aligned
    ((3, 4, 5, 48), 9, 45, "B11D", 4),       # 8-byte vectors, 9 lanes per row
    ((4, 6, 3, 96), 9, 83, "BSND", 6),       # x 4-byte / 8-byte aligned, cos/sin per head
    ((2, 5, 3, 64), 1, 63, "BS1D", 1),       # x only element-aligned: the element path
]


def odd_path(shape, start, off, dtype):
    """4 when some 16- or 8-byte vector that divides x's address (buffer base
    + off elements) and its row pitch puts the start at element 1 of a
    vector, else 2."""
    e = synth.ELEM_BYTES[dtype]
    for v in (16, 8):
        if (off * e) % v == 0 and (shape[3] * e) % v == 0 and start % (v // e) == 1:
            return 4
    return 2


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("k", range(len(ODD_STARTS)))
def test_odd_starts(dtype, k):
    """Odd starts, bit for bit against the oracle, with 4 KiB canaries on
    both sides of x that must stay unchanged."""
    shape, st, en, form, off = ODD_STARTS[k]
    x, r1, r2, g = synth.case(shape, st, en, dtype, form, seed=1500 + k)
    e = synth.ELEM_BYTES[dtype]
    guard, n = 4096 // e, x.size
    canary = np.full(guard * 2 + off + n, 0x5A5A5A5A if e == 4 else 0x5A5A,
                     dtype=np.uint32 if e == 4 else np.uint16)
    canary = canary.view(np.float32) if dtype == "fp32" else canary
    buf = to_dev(canary, dtype)
    c, s = to_dev(r1, dtype), to_dev(r2, dtype)
    lo = guard + off
    view = buf[lo:lo + n].view(shape)
    plan = binding.rope_partial_plan(view, c, s, st, en)
    assert plan.path == odd_path(shape, st, off, dtype), (plan.path, plan.vec_bytes)
    for direction, inp in (("fwd", x), ("bwd", g)):
        view.copy_(synth.to_torch(inp, dtype).to(DEV))
        fn = binding.rope_partial_inplace_fwd if direction == "fwd" else binding.rope_partial_inplace_bwd
        fn(view, c, s, st, en)
        torch.cuda.synchronize()
        host = synth.from_torch(buf)
        assert_same(host[lo:lo + n].reshape(shape), run_oracle(direction, inp, r1, r2, dtype, st, en),
                    dtype, f"{shape} [{st},{en}) {form} offset {off} {direction}")
        assert np.array_equal(host[:lo], canary[:lo]), "canary before x changed"
        assert np.array_equal(host[lo + n:], canary[lo + n:]), "canary after x changed"


# The odd-start cases bench.py times, at full size and with its inputs: the
# gqa shape (fp16, one cos/sin row per position) and the large fp32 shape
# (per-batch position offsets), each with the path and vector width the
# planner picks; every element compared, forward and backward.
ODD_FULL = [("gqa", 1, 65, 4, 16), ("gqa", 1, 63, 4, 16), ("gqa", 5, 69, 4, 8), ("gqa", 3, 45, 2, 4),
            ("large_unaligned", 1, 65, 4, 16), ("large_unaligned", 3, 67, 4, 8)]


@pytest.mark.parametrize("name,st,en,path,vec", ODD_FULL)
def test_odd_start_full_size(name, st, en, path, vec):
    w = synth.WORKLOADS[name]
    x = synth.normal(w.shape, w.dtype, w.seed)
    r1, r2 = synth.rope_table(synth.positions(w), en - st, w.dtype)
    xd, c, s = to_dev(x, w.dtype), to_dev(r1, w.dtype), to_dev(r2, w.dtype)
    plan = binding.rope_partial_plan(xd, c, s, st, en)
    assert (plan.path, plan.vec_bytes) == (path, vec)
    del xd, c, s
    for direction in ("fwd", "bwd"):
        got = run_cuda(direction, x, r1, r2, w.dtype, st, en)
        assert_same(got, run_oracle(direction, x, r1, r2, w.dtype, st, en), w.dtype,
                    f"{name} [{st},{en}) {direction}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("elem_offset", [0, 1, 2, 4])
def test_guard_bands_and_misaligned_base(dtype, elem_offset):
    """x sits inside a larger buffer, possibly only element-aligned; 4 KiB
    canaries on both sides must stay bit-unchanged."""
    shape, st, en = (3, 11, 5, 40), 4, 36
    x, r1, r2, g = synth.case(shape, st, en, dtype, "BS1D", seed=7)
    e = synth.ELEM_BYTES[dtype]
    guard = 4096 // e
    n = x.size
    canary = np.full(guard * 2 + elem_offset + n, 0x5A5A5A5A if e == 4 else 0x5A5A,
                     dtype=np.uint32 if e == 4 else np.uint16)
    canary = canary.view(np.float32) if dtype == "fp32" else canary
    buf = to_dev(canary, dtype)
    c, s = to_dev(r1, dtype), to_dev(r2, dtype)
    for direction, inp in (("fwd", x), ("bwd", g)):
        lo = guard + elem_offset
        view = buf[lo:lo + n].view(shape)
        view.copy_(synth.to_torch(inp, dtype).to(DEV))
        fn = binding.rope_partial_inplace_fwd if direction == "fwd" else binding.rope_partial_inplace_bwd
        fn(view, c, s, st, en)
        torch.cuda.synchronize()
        host = synth.from_torch(buf)
        assert_same(host[lo:lo + n].reshape(shape), run_oracle(direction, inp, r1, r2, dtype, st, en),
                    dtype, f"offset {elem_offset} {direction}")
        assert np.array_equal(host[:lo], canary[:lo]), "canary before x changed"
        assert np.array_equal(host[lo + n:], canary[lo + n:]), "canary after x changed"


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_special_values(dtype):
    """inf, nan, signed zeros, subnormals and values that overflow fp16."""
    shape, st, en = (2, 4, 3, 32), 0, 32
    rng = np.random.default_rng(5)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-40, -3e-39, 6e4, -6.5e4, 3e38,
                         1e-8, 7e-6, 65504.0, 2.0**-24, 1.0, -1.0], np.float64)
    xv = rng.choice(specials, size=shape)
    cv = rng.choice(np.array([0.0, -0.0, 1.0, 0.5, -0.75, 1e-30, 2.0, np.inf]), size=(1, 4, 1, 32))
    sv = rng.choice(np.array([0.0, 1.0, -1.0, 0.25, 3.0, 1e-20, -0.0]), size=(1, 4, 1, 32))
    with np.errstate(over="ignore", invalid="ignore"):
        x = synth.to_storage(xv, dtype)
        c = synth.to_storage(cv, dtype)
        s = synth.to_storage(sv, dtype)
    for direction in ("fwd", "bwd"):
        got = run_cuda(direction, x, c, s, dtype, st, en)
        want = run_oracle(direction, x, c, s, dtype, st, en)
        assert_same(got, want, dtype, f"specials {direction}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noops_leave_memory_untouched(dtype):
    x, r1, r2, _ = synth.case((2, 3, 4, 16), 0, 8, dtype, "BS1D", seed=3)
    xd = to_dev(x, dtype)
    empty = torch.empty((1, 1, 1, 0), dtype=xd.dtype, device=DEV)
    binding.rope_partial_inplace_fwd(xd, empty, empty, 6, 6)
    binding.rope_partial_inplace_bwd(xd, empty, empty, 0, 0)
    torch.cuda.synchronize()
    assert_same(synth.from_torch(xd), x, dtype, "start == end")
    e = torch.empty((0, 3, 4, 16), dtype=xd.dtype, device=DEV)
    c = to_dev(r1[:1], dtype)  # batch dim 1 broadcasts against B == 0
    binding.rope_partial_inplace_fwd(e, c, c, 0, 8)
    binding.rope_partial_inplace_bwd(e, c, c, 0, 8)
    torch.cuda.synchronize()


def test_side_stream_and_strided_tables():
    """A non-default stream; cos/sin as strided views of a bigger table
    (rows [5, 5 + S) of a 64-position table) and as stride-0 expansions."""
    dtype = "fp16"
    shape, st, en = (3, 17, 6, 96), 16, 80
    L = en - st
    x, _, _, _ = synth.case(shape, st, en, dtype, "BS1D", seed=11)
    pos = np.arange(64, dtype=np.int64).reshape(1, 64, 1)
    tc, ts = synth.rope_table(pos, L, dtype)                        # (1, 64, 1, L)
    big_c, big_s = to_dev(tc, dtype), to_dev(ts, dtype)
    c_view = big_c[:, 5:5 + shape[1]].expand(shape[0], shape[1], 1, L)  # B via stride 0
    s_view = big_s[:, 5:5 + shape[1]].expand(shape[0], shape[1], 1, L)
    assert c_view.stride()[0] == 0
    side = torch.cuda.Stream()
    xd = to_dev(x, dtype)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        binding.rope_partial_inplace_fwd(xd, c_view, s_view, st, en)
    side.synchronize()
    want = oracle.fwd(x, np.ascontiguousarray(tc[:, 5:5 + shape[1]]),
                      np.ascontiguousarray(ts[:, 5:5 + shape[1]]), dtype, st, en)
    assert_same(synth.from_torch(xd), want, dtype, "strided tables on a side stream")


def test_round_trip_fp32():
    """bwd(fwd(x)) returns x within 1e-6 of each pair's norm for a cos/sin table."""
    w = synth.WORKLOADS["large_unaligned"]
    shape = (1, 2048, 32, 128)
    x = synth.normal(shape, "fp32", 1)
    pos = synth.positions(w)[:1, :2048]
    c, s = synth.rope_table(pos, w.L, "fp32")
    xd, cd, sd = to_dev(x, "fp32"), to_dev(c, "fp32"), to_dev(s, "fp32")
    binding.rope_partial_inplace_fwd(xd, cd, sd, w.start, w.end)
    binding.rope_partial_inplace_bwd(xd, cd, sd, w.start, w.end)
    back = synth.from_torch(xd).astype(np.float64)
    xs = x[..., w.start:w.end].astype(np.float64)
    norm = np.repeat(np.sqrt(xs[..., 0::2] ** 2 + xs[..., 1::2] ** 2), 2, axis=-1)
    assert (np.abs(back[..., w.start:w.end] - xs) / norm).max() <= 1e-6
    assert np.array_equal(back[..., :w.start], x[..., :w.start].astype(np.float64))


@pytest.mark.parametrize("shape,launches", [((2, 2**30 + 3, 1, 2), 2), ((1, 2**31 + 5, 1, 2), 2)])
def test_calls_split_into_several_launches(shape, launches):
    """8.6 GB fp16 tensors with one pair per row: more than 2^31 work items,
    so the call runs as several launches.  With cos = 0 and sin = 1 the
    forward is the exact quarter turn (a, b) -> (-b, a), a property that
    holds at any size; rows next to the launch boundaries are also checked
    against the oracle one by one."""
    B, S, N, D = shape
    g = torch.Generator(device=DEV).manual_seed(1234)
    x = torch.randn(shape, generator=g, device=DEV, dtype=torch.float32).to(torch.float16)
    zero = torch.zeros((1, 1, 1, 2), dtype=torch.float16, device=DEV)
    one = torch.ones((1, 1, 1, 2), dtype=torch.float16, device=DEV)
    plan = binding.rope_partial_plan(x, zero, one, 0, 2)
    assert plan.launches == launches
    ref = x.clone()
    binding.rope_partial_inplace_fwd(x, zero, one, 0, 2)
    torch.cuda.synchronize()
    assert torch.equal(x[..., 0], -ref[..., 1]) and torch.equal(x[..., 1], ref[..., 0])
    # rows around each boundary, through the oracle, with a random table
    c_h, s_h = synth.random_table((1, 1, 1, 2), "fp16", 9)
    x2 = ref.clone()
    binding.rope_partial_inplace_fwd(x2, to_dev(c_h, "fp16"), to_dev(s_h, "fp16"), 0, 2)
    torch.cuda.synchronize()
    flat_in, flat_out = ref.view(-1, 2), x2.view(-1, 2)
    T = B * S
    for t0 in (0, 2**31 - 2, S - 2 if B > 1 else 2**31 - 4, T - 3):
        rows_in = synth.from_torch(flat_in[t0:t0 + 3]).reshape(1, 3, 1, 2)
        rows_out = synth.from_torch(flat_out[t0:t0 + 3]).reshape(1, 3, 1, 2)
        assert_same(rows_out, oracle.fwd(rows_in, c_h, s_h, "fp16", 0, 2), "fp16", f"rows at {t0}")
    del x, x2, ref
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_tables_packed_right_after_x(dtype):
    """x, cos and sin packed back to back in one allocation (adjacent byte
    ranges that do not overlap) are accepted and rotate as separate tensors
    would; the overlap rule refuses only shared bytes."""
    shape, st, en = (2, 5, 3, 32), 2, 30
    x, r1, r2, g = synth.case(shape, st, en, dtype, "BS1D", seed=21)
    td = synth.TORCH_DTYPE[dtype]
    n, m = x.size, r1.size
    buf = torch.empty(n + 2 * m, dtype=td, device=DEV)
    xv, cv, sv = buf[:n].view(shape), buf[n:n + m].view(r1.shape), buf[n + m:].view(r2.shape)
    cv.copy_(synth.to_torch(r1, dtype).to(DEV))
    sv.copy_(synth.to_torch(r2, dtype).to(DEV))
    for direction, inp in (("fwd", x), ("bwd", g)):
        xv.copy_(synth.to_torch(inp, dtype).to(DEV))
        fn = binding.rope_partial_inplace_fwd if direction == "fwd" else binding.rope_partial_inplace_bwd
        fn(xv, cv, sv, st, en)
        torch.cuda.synchronize()
        assert_same(synth.from_torch(xv), run_oracle(direction, inp, r1, r2, dtype, st, en), dtype,
                    f"packed {direction}")
        assert np.array_equal(synth.from_torch(cv).view(np.uint8), r1.view(np.uint8))
        assert np.array_equal(synth.from_torch(sv).view(np.uint8), r2.view(np.uint8))

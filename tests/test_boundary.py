"""The C ABI without a GPU: exports, validation, empty calls and launch plans.

Every call here is rejected or empty (returns before any CUDA call), or is a
plan query with an explicit SM count, so nothing touches a device.  Fake
pointers are plain aligned integers and are never dereferenced.

The rules follow "CANN ops-transformer inplace_partial_rotary_mul", section
约束说明 (D even and <= 1024; 0 <= start <= end <= D with an even length;
r1/r2 broadcast against the slice with last dim end - start; one dtype),
and section 功能与计算公式 (start == end is a no-op; the backward accepts
empty tensors).
"""
import ctypes
import os
import re
import subprocess

import pytest

from place_partial_rope_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rope_partial.h")
OK, NULLPTR, INVALID, CUDA = 0, 1, 2, 3
BF16, FP16, FP32 = 0, 1, 2
BASE = 0x7F0000000000  # a fake, 256-byte aligned device address


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def i64(*v):
    return (ctypes.c_int64 * 4)(*v)


def contig(shape):
    B, S, N, L = shape
    return (S * N * L, N * L, L, 1)


def call(lib, fn="rope_partial_inplace_fwd", x=BASE, r1=BASE + 2**30, r2=BASE + 2**31,
         dtype=FP16, shape=(2, 4, 3, 16), start=0, end=8, r_shape=None, r_stride=None,
         r2_shape=None, r2_stride=None):
    B, S, N, D = shape
    rs = r_shape if r_shape is not None else (1, S, 1, end - start)
    rst = r_stride if r_stride is not None else (contig(rs) if rs != "null" else (0, 0, 0, 1))
    r2s = r2_shape if r2_shape is not None else rs
    r2st = r2_stride if r2_stride is not None else (contig(r2s) if r2s != "null" else (0, 0, 0, 1))
    a1 = i64(*rs) if rs != "null" else None
    a2 = i64(*rst) if rst != "null" else None
    a3 = i64(*r2s) if r2s != "null" else None
    a4 = i64(*r2st) if r2st != "null" else None
    return getattr(lib, fn)(x, r1, r2, dtype, B, S, N, D, a1, a2, a3, a4, start, end, None)


def test_header_symbols_are_exported(lib):
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(rope_[a-z_]+)\s*\(", text))
    assert names == {"rope_partial_inplace_fwd", "rope_partial_inplace_bwd",
                     "rope_partial_inplace_fwd_host", "rope_partial_inplace_bwd_host",
                     "rope_partial_inplace_fwd_qk", "rope_partial_inplace_bwd_qk",
                     "rope_partial_inplace_fwd_mode", "rope_partial_inplace_bwd_mode",
                     "rope_partial_inplace_fwd_pos", "rope_partial_inplace_bwd_pos",
                     "rope_partial_plan_mode", "rope_partial_token_shard",
                     "rope_status_str", "rope_last_error_message", "rope_partial_plan"}
    for n in names:
        assert hasattr(lib, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                        capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (rope_\w+)", nm))
    assert names <= exported


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load_library()


def test_status_strings(lib):
    assert lib.rope_status_str(OK) == b"ROPE_OK"
    assert lib.rope_status_str(INVALID) == b"ROPE_ERR_INVALID"
    assert lib.rope_status_str(CUDA) == b"ROPE_ERR_CUDA"
    assert lib.rope_status_str(99) == b"ROPE_ERR_UNKNOWN"


ALL_FNS = ["rope_partial_inplace_fwd", "rope_partial_inplace_bwd", "rope_partial_inplace_fwd_host",
           "rope_partial_inplace_bwd_host"]


@pytest.mark.parametrize("fn", ALL_FNS)
@pytest.mark.parametrize("kwargs,status,needle", [
    (dict(dtype=3), INVALID, "dtype"),
    (dict(dtype=-1), INVALID, "dtype"),
    (dict(shape=(-1, 4, 3, 16)), INVALID, "negative"),
    (dict(shape=(2, 4, 3, 15), end=8), INVALID, "even"),
    (dict(shape=(1, 1, 1, 1026), end=2), INVALID, "1024"),
    (dict(start=-2, end=4), INVALID, "slice"),
    (dict(start=10, end=8), INVALID, "slice"),
    (dict(start=0, end=18), INVALID, "slice"),
    (dict(start=1, end=8), INVALID, "even"),
    (dict(r_shape=(1, 3, 1, 8)), INVALID, "broadcast"),
    (dict(r_shape=(2, 4, 2, 8)), INVALID, "broadcast"),
    (dict(r_shape=(1, 4, 1, 6)), INVALID, "last dim"),
    (dict(r2_shape=(1, 4, 1, 4)), INVALID, "r2 last dim"),
    (dict(r_stride=(32, 8, 8, 2)), INVALID, "contiguous"),
    (dict(r_stride=(32, -8, 8, 1)), INVALID, "negative"),
    (dict(x=0), NULLPTR, "x is null"),
    (dict(r1=0), NULLPTR, "r1"),
    (dict(r2=0), NULLPTR, "r2"),
    (dict(r_shape="null"), NULLPTR, "r1_shape"),
    (dict(r2_stride="null"), NULLPTR, "r2_stride"),
    (dict(x=BASE + 1), INVALID, "aligned"),
    (dict(dtype=FP32, x=BASE + 2), INVALID, "aligned"),
    (dict(r1=BASE + 3), INVALID, "aligned"),
])
def test_rejected_calls(lib, fn, kwargs, status, needle):
    st = call(lib, fn, **kwargs)
    assert st == status, (st, lib.rope_last_error_message())
    assert needle in lib.rope_last_error_message().decode()


@pytest.mark.parametrize("fn", ALL_FNS)
@pytest.mark.parametrize("kwargs", [
    dict(start=4, end=4, x=0, r1=0, r2=0),                      # empty slice, null pointers
    dict(start=0, end=0, x=0, r1=0, r2=0, r_shape="null", r2_shape="null",
         r_stride="null", r2_stride="null"),                    # nothing at all
    dict(shape=(0, 4, 3, 16), x=0, r1=0, r2=0, r_shape=(1, 4, 1, 8)),   # B == 0
    dict(shape=(2, 0, 3, 16), r_shape=(1, 0, 1, 8)),            # S == 0
    dict(shape=(2, 4, 0, 16), r_shape=(1, 4, 1, 8)),            # N == 0
    dict(shape=(2, 4, 3, 0), start=0, end=0, r_shape=(1, 4, 1, 0)),  # D == 0
])
def test_empty_calls_are_noops(lib, fn, kwargs):
    assert call(lib, fn, **kwargs) == OK, lib.rope_last_error_message()


def plan(lib, x=BASE, r1=BASE + 2**30, r2=BASE + 2**31, dtype=FP16, shape=(2, 4, 3, 16),
         start=0, end=8, r_shape=None, r_stride=None, sms=152):
    B, S, N, D = shape
    rs = r_shape or (1, S, 1, end - start)
    rst = r_stride or contig(rs)
    p = binding.RopePlan()
    st = lib.rope_partial_plan(x, r1, r2, dtype, B, S, N, D, i64(*rs), i64(*rst), i64(*rs),
                               i64(*rst), start, end, sms, ctypes.byref(p))
    assert st == OK, lib.rope_last_error_message()
    return p


def test_plans_of_the_named_workloads(lib):
    # GQA fp16: 128-byte slices at offset 0 of 256-byte rows -> 16-byte accesses
    p = plan(lib, dtype=FP16, shape=(32, 2048, 16, 128), start=0, end=64, r_shape=(1, 2048, 1, 64))
    assert (p.path, p.vec_bytes, p.chunks_per_row, p.heads_per_thread, p.r_per_head) == (1, 16, 8, 4, 0)
    # 16-bit interleave: one block per 256 work items
    assert p.tasks == 32 * 2048 * 4 * 8 and p.blocks == p.tasks // 256 and p.launches == 1
    # MLA-decode query bf16: one cos/sin row per token
    p = plan(lib, dtype=BF16, shape=(4096, 1, 128, 192), start=0, end=64, r_shape=(4096, 1, 1, 64))
    assert (p.path, p.vec_bytes, p.chunks_per_row, p.heads_per_thread) == (1, 16, 8, 4)
    # large fp32 with the slice at byte 136: 8-byte accesses hold whole pairs
    p = plan(lib, dtype=FP32, shape=(4, 8192, 32, 128), start=34, end=98, r_shape=(4, 8192, 1, 64))
    assert (p.path, p.vec_bytes, p.chunks_per_row, p.heads_per_thread) == (1, 8, 32, 4)
    assert p.blocks == p.tasks // 256  # one block per 256 work items
    # tiny fp32 (16-byte accesses: 2 heads per thread) and the small-model
    # bf16 full-row slice
    p = plan(lib, dtype=FP32, shape=(1, 16, 2, 64), start=0, end=32, r_shape=(1, 16, 1, 32))
    assert (p.path, p.vec_bytes, p.heads_per_thread, p.blocks) == (1, 16, 2, 1)
    p = plan(lib, dtype=BF16, shape=(16, 256, 12, 64), start=0, end=64, r_shape=(1, 256, 1, 64))
    assert (p.path, p.vec_bytes, p.heads_per_thread) == (1, 16, 4)


def test_path_choice(lib):
    ODD = 4
    # odd start at element 1 of an aligned 16- or 8-byte vector of x (the
    # widest that divides x's address and its row pitch): a lane per vector
    p = plan(lib, start=1, end=9)                                     # 4 pairs in one lane
    assert (p.path, p.vec_bytes, p.chunks_per_row, p.heads_per_thread) == (ODD, 16, 1, 2)
    p = plan(lib, dtype=FP16, shape=(32, 2048, 16, 128), start=1, end=65, r_shape=(1, 2048, 1, 64))
    assert (p.path, p.vec_bytes, p.chunks_per_row, p.heads_per_thread) == (ODD, 16, 8, 4)
    assert p.blocks == p.tasks // 256
    p = plan(lib, dtype=FP16, shape=(32, 2048, 16, 128), start=1, end=63, r_shape=(1, 2048, 1, 62))
    assert (p.path, p.vec_bytes, p.chunks_per_row) == (ODD, 16, 8)   # 31 pairs: last lane partial
    p = plan(lib, dtype=FP16, shape=(2, 4, 3, 64), start=9, end=51, r_shape=(1, 4, 1, 42))
    assert (p.path, p.vec_bytes, p.chunks_per_row) == (ODD, 16, 6)    # 21 pairs
    p = plan(lib, shape=(2, 4, 3, 16), start=1, end=7, r_shape=(1, 4, 1, 6))
    assert (p.path, p.vec_bytes, p.chunks_per_row) == (ODD, 16, 1)    # 3 pairs
    p = plan(lib, start=1, end=9, x=BASE + 8)                         # x only 8-byte aligned
    assert (p.path, p.vec_bytes, p.chunks_per_row, p.heads_per_thread) == (ODD, 8, 2, 2)
    p = plan(lib, dtype=FP32, start=1, end=9)                         # fp32: 2 pairs per lane
    assert (p.path, p.vec_bytes, p.chunks_per_row) == (ODD, 16, 2)
    p = plan(lib, dtype=FP32, start=1, end=9, x=BASE + 8)             # fp32: 1 pair per lane
    assert (p.path, p.vec_bytes, p.chunks_per_row) == (ODD, 8, 4)
    # no 16-byte vector starts at element 1, an 8-byte one does
    p = plan(lib, start=5, end=13)                                    # element 5 of 8, 1 of 4
    assert (p.path, p.vec_bytes, p.chunks_per_row) == (ODD, 8, 2)
    p = plan(lib, dtype=FP32, start=3, end=11)                        # fp32: any odd start at 8 bytes
    assert (p.path, p.vec_bytes, p.chunks_per_row) == (ODD, 8, 4)
    # other odd starts take the element path
    assert plan(lib, start=3, end=11).path == 2                      # element 3 of 8 and of 4
    assert plan(lib, start=1, end=9, x=BASE + 4).path == 2           # x only 4-byte aligned
    assert plan(lib, shape=(2, 4, 3, 18), start=1, end=9).path == 2  # 36-byte rows
    assert plan(lib, start=1, end=9, x=BASE + 2).path == 2           # x only 2-byte aligned
    assert plan(lib, start=1, end=9, r1=BASE + 2**30 + 2).path == 2  # cos only 2-byte aligned
    assert plan(lib, dtype=FP32, start=1, end=9, x=BASE + 4).path == 2   # fp32 needs 8 bytes
    assert plan(lib, start=2, end=10).vec_bytes == 4                 # 4-byte slice offset
    assert plan(lib, x=BASE + 8).vec_bytes == 8                      # x only 8-byte aligned
    assert plan(lib, r1=BASE + 2**30 + 4).vec_bytes == 4             # cos only 4-byte aligned
    assert plan(lib, dtype=FP32, x=BASE + 4).path == 2               # fp32 pairs need 8 bytes
    assert plan(lib, shape=(2, 4, 3, 18), end=8).vec_bytes == 4      # 36-byte rows
    p = plan(lib, r_shape=(2, 4, 3, 8))                               # cos/sin per head (BSND)
    assert p.r_per_head == 1
    assert plan(lib, r_shape=(1, 4, 3, 8)).r_per_head == 1           # 1SND
    assert plan(lib, r_shape=(2, 1, 1, 8)).r_per_head == 0           # B11D


@pytest.mark.parametrize("N,vec,U", [(1, 16, 1), (2, 16, 2), (3, 16, 2), (5, 16, 2), (7, 16, 4),
                                     (12, 16, 4), (16, 16, 4), (12, 8, 2), (32, 8, 2), (6, 8, 2),
                                     (5, 8, 2)])
def test_heads_per_thread(lib, N, vec, U):
    """16-bit rows: up to 4 heads per thread for 16-byte chunks, 2 for 8-byte
    chunks, never more than a quarter of the head slots idle."""
    start = 0 if vec == 16 else 4  # 8-byte slice offset forces 8-byte accesses for fp16
    p = plan(lib, shape=(1, 2, N, 64), start=start, end=start + 48, r_shape=(1, 2, 1, 48))
    assert p.vec_bytes == vec and p.heads_per_thread == U


@pytest.mark.parametrize("start,end,chunks,U", [(0, 16, 2, 1), (0, 32, 4, 2), (16, 48, 4, 2),
                                                (0, 48, 6, 4), (0, 64, 8, 4)])
def test_heads_per_thread_short_16bit_slices(lib, start, end, chunks, U):
    """16-byte accesses of a short 16-bit slice: one head per thread for 2
    accesses per row, two for 4, four from 6 on; half-split rows whose
    accesses fit a warp take one for 2 and four otherwise."""
    p = plan(lib, shape=(32, 64, 16, 128), start=start, end=end, r_shape=(1, 64, 1, end - start))
    assert (p.vec_bytes, p.chunks_per_row, p.heads_per_thread) == (16, chunks, U)
    st, p = plan_mode(lib, 2, shape=(32, 64, 16, 128), start=start, end=end,
                      r_shape=(1, 64, 1, end - start))
    assert st == OK and p.heads_per_thread == (1 if chunks <= 2 else 4)


@pytest.mark.parametrize("start,end,mode,vec,U", [
    (32, 96, 1, 16, 2),    # fp32 16-byte accesses: 32 bytes of x per thread
    (34, 98, 1, 8, 4),     # 8-byte accesses
    (1, 65, 1, 16, 4),     # odd start: a lane per aligned 16-byte vector (4 heads)
    (34, 98, 2, 8, 4),     # half-split, partner in another lane (32 accesses per row)
    (0, 96, 2, 16, 2),     # half-split, 48 lanes per half = 12 accesses: both halves in one thread
    (2, 98, 2, 8, 2),      # 24 accesses per half of 8 bytes: both halves in one thread
])
def test_heads_per_thread_fp32(lib, start, end, mode, vec, U):
    """fp32 rows: about 32 bytes of x per thread (a thread that holds both
    halves of a half-split pair counts both accesses)."""
    st, p = plan_mode(lib, mode, dtype=FP32, shape=(4, 64, 32, 128), start=start, end=end,
                      r_shape=(4, 64, 1, end - start))
    assert st == OK and (p.vec_bytes, p.heads_per_thread) == (vec, U)
    assert p.blocks == -(-p.tasks // 256)  # one block per 256 work items


def test_huge_calls_split_into_launches(lib):
    # fp16 rows of 2 elements, one head: one work item per token
    p = plan(lib, shape=(2, 2**30 + 3, 1, 2), start=0, end=2, r_shape=(1, 2**30 + 3, 1, 2))
    assert p.launches == 2 and p.tasks == 2 * (2**30 + 3)            # whole batches per launch
    p = plan(lib, shape=(1, 2**31 + 5, 1, 2), start=0, end=2, r_shape=(1, 2**31 + 5, 1, 2))
    assert p.launches == 2                                           # runs of tokens of one batch
    p = plan(lib, shape=(3, 2**31 + 5, 1, 2), start=0, end=2, r_shape=(1, 2**31 + 5, 1, 2))
    assert p.launches == 6
    p = plan(lib, shape=(2**20, 2**11, 1, 2), start=0, end=2, r_shape=(1, 2**11, 1, 2))
    assert p.launches == 1                                           # exactly 2^31 items
    # the odd-start kernel (one lane per row for 4 pairs) splits the same way
    p = plan(lib, shape=(2, 2**30 + 3, 1, 16), start=1, end=9, r_shape=(1, 2**30 + 3, 1, 8))
    assert (p.path, p.launches, p.tasks) == (4, 2, 2 * (2**30 + 3))


def test_fast_division_exhaustive_sample(tmp_path):
    """The multiply-high division used by the kernels, against / and %."""
    src = tmp_path / "t.cpp"
    src.write_text(r'''
#include "fast_div.h"
#include <cstdio>
#include <cstdint>
int main() {
  uint64_t bad = 0, n_checked = 0;
  uint32_t divs[] = {1u,2u,3u,5u,7u,8u,12u,31u,32u,64u,96u,128u,255u,1000u,2048u,4095u,65537u,
                     (1u<<20)+7u,(1u<<30)+3u,(1u<<31)-1u,(1u<<31),(1u<<31)+1u,4294967295u};
  for (uint32_t d : divs) {
    rope::FastDiv f = rope::FastDiv::make(d);
    for (uint64_t n = 0; n < (1ull<<32); n += 0x10001ull + d) {
      uint32_t q, r; f.divmod((uint32_t)n, q, r); ++n_checked;
      if (q != (uint32_t)n / d || r != (uint32_t)n % d) ++bad;
    }
    for (uint64_t k = 0; k < 4096; ++k) {
      uint32_t n = 0xffffffffu - (uint32_t)k, q, r; f.divmod(n, q, r); ++n_checked;
      if (q != n / d || r != n % d) ++bad;
      n = (uint32_t)k * d; f.divmod(n, q, r); if (q != n / d || r != n % d) ++bad;
      if (n) { --n; f.divmod(n, q, r); if (q != n / d || r != n % d) ++bad; }
    }
  }
  std::printf("%llu %llu\n", (unsigned long long)bad, (unsigned long long)n_checked);
  return bad != 0;
}
''')
    exe = tmp_path / "t"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", os.path.join(build.CSRC), str(src), "-o",
                    str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout


def qk_call(lib, fn="rope_partial_inplace_fwd_qk", q=BASE, k=BASE + 2**32, r1=BASE + 2**30,
            r2=BASE + 2**31, dtype=BF16, B=4, S=1, Nq=8, Dq=192, qs=0, qe=64, Nk=1, Dk=64, ks=0,
            ke=64, r_shape=None):
    rs = r_shape or (B, S, 1, qe - qs)
    rst = contig(rs)
    return getattr(lib, fn)(q, k, r1, r2, dtype, B, S, Nq, Dq, qs, qe, Nk, Dk, ks, ke,
                            i64(*rs), i64(*rst), i64(*rs), i64(*rst), None)


@pytest.mark.parametrize("fn", ["rope_partial_inplace_fwd_qk", "rope_partial_inplace_bwd_qk"])
@pytest.mark.parametrize("kwargs,status,needle", [
    (dict(ks=0, ke=32), INVALID, "differ"),                 # slice lengths differ
    (dict(r_shape=(4, 1, 8, 64)), INVALID, "head dim"),     # per-head cos/sin not shared
    (dict(Dq=191), INVALID, "query"),                       # query: odd head dim
    (dict(Dk=66, ks=4, ke=68 + 2), INVALID, "key"),         # key: slice end beyond its D
    (dict(k=0), NULLPTR, "key"),
    (dict(q=BASE + 1), INVALID, "query"),
])
def test_qk_rejected_calls(lib, fn, kwargs, status, needle):
    st = qk_call(lib, fn, **kwargs)
    assert st == status, (st, lib.rope_last_error_message())
    assert needle in lib.rope_last_error_message().decode()


@pytest.mark.parametrize("fn", ALL_FNS)
@pytest.mark.parametrize("kwargs,needle", [
    (dict(r1=BASE + 16), "r1 (cos) overlaps x"),             # cos inside x
    (dict(r2=BASE + 766), "r2 (sin) overlaps x"),            # sin's first bytes on x's last
    (dict(r1=BASE - 62), "r1 (cos) overlaps x"),             # cos's last row runs into x
])
def test_cos_sin_overlapping_x_are_rejected(lib, fn, kwargs, needle):
    """x is written in place while r1 and r2 are read, so a call whose x
    shares a byte with either is refused before any CUDA call (x here is
    2*4*3*16 fp16 = 768 bytes; cos/sin (1, 4, 1, 8) span 64 bytes)."""
    st = call(lib, fn, **kwargs)
    assert st == INVALID, (st, lib.rope_last_error_message())
    assert needle in lib.rope_last_error_message().decode()


@pytest.mark.parametrize("fn", ["rope_partial_inplace_fwd_qk", "rope_partial_inplace_bwd_qk"])
@pytest.mark.parametrize("kwargs,needle", [
    (dict(k=BASE + 4 * 8 * 192 * 2 - 2), "query and key overlap"),   # key starts on q's last element
    (dict(k=BASE + 64), "query and key overlap"),
    (dict(r1=BASE + 2**32 + 32), "overlaps the key"),
    (dict(r2=BASE + 1024), "overlaps the query"),
])
def test_qk_overlapping_tensors_are_rejected(lib, fn, kwargs, needle):
    st = qk_call(lib, fn, **kwargs)
    assert st == INVALID, (st, lib.rope_last_error_message())
    assert needle in lib.rope_last_error_message().decode()


def test_qk_empty_calls(lib):
    assert qk_call(lib, qs=0, qe=0, ks=5, ke=5, q=0, k=0, r1=0, r2=0) == OK   # empty slices
    assert qk_call(lib, B=0, q=0, k=0, r1=0, r2=0, r_shape=(1, 1, 1, 64)) == OK


def plan_mode(lib, mode, x=BASE, r1=BASE + 2**30, r2=BASE + 2**31, dtype=FP16, shape=(2, 4, 3, 16),
              start=0, end=8, r_shape=None):
    B, S, N, D = shape
    rs = r_shape or (1, S, 1, end - start)
    rst = contig(rs)
    p = binding.RopePlan()
    st = lib.rope_partial_plan_mode(x, r1, r2, dtype, B, S, N, D, i64(*rs), i64(*rst), i64(*rs),
                                    i64(*rst), start, end, mode, 152, ctypes.byref(p))
    return st, p


def test_half_split_plans(lib):
    HALF, LANES = 2, 3
    # gqa-like fp16: the 64-lane slice is 8 accesses of 16 bytes, one warp's
    # worth, so the partner access (4 lanes on) comes by shuffle; 4 heads per
    # thread and one block per 256 items, as in interleave mode
    st, p = plan_mode(lib, HALF, shape=(32, 2048, 16, 128), start=0, end=64, r_shape=(1, 2048, 1, 64))
    assert st == OK and (p.path, p.vec_bytes, p.chunks_per_row, p.heads_per_thread) == (LANES, 16, 8, 4)
    assert p.blocks == p.tasks // 256
    # fp32 slice at byte 136: 8-byte accesses (each half is 128 bytes), 32 per row
    st, p = plan_mode(lib, HALF, dtype=FP32, shape=(4, 8192, 32, 128), start=34, end=98,
                      r_shape=(4, 8192, 1, 64))
    assert st == OK and (p.path, p.vec_bytes, p.chunks_per_row, p.heads_per_thread) == (LANES, 8, 32, 4)
    assert p.blocks == p.tasks // 256
    # fp16 odd start: single elements, both halves in one thread
    st, p = plan_mode(lib, HALF, start=1, end=9)
    assert st == OK and (p.path, p.vec_bytes, p.chunks_per_row) == (2, 2, 4)
    # fp32 odd start: a 4-byte access is one element; 8 per row
    st, p = plan_mode(lib, HALF, dtype=FP32, start=1, end=9)
    assert st == OK and (p.path, p.vec_bytes, p.chunks_per_row) == (LANES, 4, 8)
    # half of L = 2 lanes of fp16 is 4 bytes: 2 accesses per row
    st, p = plan_mode(lib, HALF, start=0, end=4)
    assert st == OK and (p.path, p.vec_bytes, p.chunks_per_row) == (LANES, 4, 2)
    # 6 accesses per row (not a power of two): both halves in one thread
    st, p = plan_mode(lib, HALF, shape=(2, 4, 3, 64), start=0, end=48)
    assert st == OK and (p.path, p.vec_bytes, p.chunks_per_row) == (1, 16, 3)
    # 128 accesses per row (more than a warp): both halves in one thread,
    # 64 accesses of the first half
    st, p = plan_mode(lib, HALF, dtype=FP32, shape=(2, 4, 3, 512), start=0, end=512)
    assert st == OK and (p.path, p.vec_bytes, p.chunks_per_row) == (1, 16, 64)
    # both halves in one thread: one block per 256 work items, 2 heads per
    # thread for fp32 16- and 8-byte accesses
    st, p = plan_mode(lib, HALF, dtype=FP32, shape=(4, 8192, 32, 128), start=0, end=96,
                      r_shape=(4, 8192, 1, 96))
    assert st == OK and (p.path, p.vec_bytes, p.heads_per_thread) == (1, 16, 2)
    assert p.blocks == p.tasks // 256
    st, p = plan_mode(lib, HALF, dtype=FP32, shape=(4, 8192, 32, 128), start=2, end=98,
                      r_shape=(4, 8192, 1, 96))
    assert st == OK and (p.path, p.vec_bytes, p.heads_per_thread) == (1, 8, 2)
    assert p.blocks == p.tasks // 256
    # 32 accesses per row: the largest that fits one warp
    st, p = plan_mode(lib, HALF, dtype=FP32, shape=(2, 4, 3, 128), start=0, end=128)
    assert st == OK and (p.path, p.vec_bytes, p.chunks_per_row) == (LANES, 16, 32)


@pytest.mark.parametrize("mode", [0, 3, -1])
def test_unknown_mode_rejected(lib, mode):
    st, _ = plan_mode(lib, mode)
    assert st == INVALID and "mode" in lib.rope_last_error_message().decode()
    B, S, N, D = 2, 4, 3, 16
    rs = (1, S, 1, 8)
    for fn in (lib.rope_partial_inplace_fwd_mode, lib.rope_partial_inplace_bwd_mode):
        st = fn(BASE, BASE + 2**30, BASE + 2**31, FP16, B, S, N, D, i64(*rs), i64(*contig(rs)),
                i64(*rs), i64(*contig(rs)), 0, 8, mode, None)
        assert st == INVALID


def pos_call(lib, fn="rope_partial_inplace_fwd_pos", x=BASE, pos=BASE + 2**30, dtype=FP16,
             shape=(2, 4, 3, 16), p_shape=(2, 4), p_stride=(4, 1), base=10000.0, start=0, end=8,
             mode=1):
    B, S, N, D = shape
    ps = (ctypes.c_int64 * 2)(*p_shape) if p_shape != "null" else None
    pst = (ctypes.c_int64 * 2)(*p_stride)
    return getattr(lib, fn)(x, pos, dtype, B, S, N, D, ps, pst, base, start, end, mode, None)


@pytest.mark.parametrize("fn", ["rope_partial_inplace_fwd_pos", "rope_partial_inplace_bwd_pos"])
@pytest.mark.parametrize("kwargs,status,needle", [
    (dict(base=0.0), INVALID, "base"),
    (dict(base=-2.0), INVALID, "base"),
    (dict(base=float("nan")), INVALID, "base"),
    (dict(base=float("inf")), INVALID, "base"),
    (dict(mode=0), INVALID, "mode"),
    (dict(pos=0), NULLPTR, "positions"),
    (dict(p_shape="null"), NULLPTR, "pos_shape"),
    (dict(p_shape=(3, 4)), INVALID, "positions dim 0"),
    (dict(p_shape=(2, 2)), INVALID, "positions dim 1"),
    (dict(p_stride=(-4, 1)), INVALID, "negative"),
    (dict(pos=BASE + 2**30 + 2), INVALID, "aligned"),
    (dict(x=0), NULLPTR, "x is null"),
    (dict(start=1, end=8), INVALID, "even"),
    (dict(shape=(2, 4, 3, 15)), INVALID, "even"),
])
def test_pos_rejected_calls(lib, fn, kwargs, status, needle):
    st = pos_call(lib, fn, **kwargs)
    assert st == status, (st, lib.rope_last_error_message())
    assert needle in lib.rope_last_error_message().decode()


def test_pos_empty_calls(lib):
    assert pos_call(lib, start=4, end=4, x=0, pos=0, p_shape="null") == OK
    assert pos_call(lib, shape=(0, 4, 3, 16), x=0, pos=0, p_shape=(1, 4)) == OK
    assert pos_call(lib, p_shape=(1, 1), p_stride=(0, 0), start=4, end=4) == OK


def test_cuda_failure_is_reported_not_raised(lib):
    """A valid plan query with sm_count = 0 asks the current device.  Without
    a usable GPU that query fails and comes back as ROPE_ERR_CUDA with a
    message; with a GPU it succeeds.  Nothing is launched either way."""
    import torch
    B, S, N, D = 2, 4, 3, 16
    rs = (1, S, 1, 8)
    p = binding.RopePlan()
    st = lib.rope_partial_plan(BASE, BASE + 2**30, BASE + 2**31, FP16, B, S, N, D, i64(*rs),
                               i64(*contig(rs)), i64(*rs), i64(*contig(rs)), 0, 8, 0,
                               ctypes.byref(p))
    if torch.cuda.is_available():
        assert st == OK and p.blocks > 0
    else:
        assert st == CUDA
        assert lib.rope_last_error_message().decode() != ""


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("dtype", [BF16, FP16, FP32])
def test_every_plan_has_a_kernel(lib, dtype, mode):
    """Sweep slice offsets, lengths, head dims, head counts and pointer
    alignments: every valid call's plan names a compiled kernel instance
    (rope_partial_plan_mode reports a missing one as ROPE_ERR_CUDA)."""
    e = 4 if dtype == FP32 else 2
    count = 0
    for D in (2, 6, 24, 64, 130, 1024):
        for start in sorted({0, 1, 2, 3, 4, 8, D // 2 - (D // 2) % 2}):
            for L in (2, 4, 6, 8, 16, 64, 1022):
                end = start + L
                if end > D:
                    continue
                for N in (1, 3, 8, 33):
                    for xoff in (0, e, 4, 8):
                        if xoff % e:
                            continue
                        st, p = plan_mode(lib, mode, x=BASE + xoff, dtype=dtype,
                                          shape=(2, 3, N, D), start=start, end=end,
                                          r_shape=(1, 3, 1, L))
                        assert st == OK, (D, start, L, N, xoff, lib.rope_last_error_message())
                        assert p.blocks > 0 and p.heads_per_thread in (1, 2, 4, 8)
                        count += 1
    assert count > 500

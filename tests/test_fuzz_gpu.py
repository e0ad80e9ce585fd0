"""Seeded random cases through every device entry point, against the oracle.

Each case draws a dtype, a head dim, a slice (odd starts, empty and full
slices included), a broadcast form for cos/sin, an element offset for x
inside a larger buffer (so its base may be only element-aligned), and
cos/sin as views into padded rows at an element offset (row strides that
are not a multiple of any access width).  The table calls, in both rotary
modes, the zero-copy calls on page-locked host buffers, and the fused
query + key call must match the oracle bit for bit,
with the canaries around x unchanged; the call that computes cos/sin from
positions must match within the bound its header states.  The draws are
fixed by the seed (tests/fuzz_cases.py); a CPU test checks that they reach
every kernel path.
"""
import numpy as np
import pytest
import torch

import fuzz_cases as fc
import oracle
from gpu_util import DEV, assert_close_pos, assert_same, to_dev
from place_partial_rope_gb300 import binding, synth

pytestmark = pytest.mark.gpu

N_TABLE, N_QK, N_POS, N_HOST = 1200, 300, 300, 300
GUARD = 64  # canary elements after x


def canary(n_elems: int, dtype: str) -> np.ndarray:
    e = synth.ELEM_BYTES[dtype]
    a = np.full(n_elems, 0x5A5A5A5A if e == 4 else 0x5A5A, np.uint32 if e == 4 else np.uint16)
    return a.view(np.float32) if dtype == "fp32" else a


def in_buffer(a: np.ndarray, offset: int, dtype: str):
    """A device buffer of canaries with `a` copied in at element `offset`;
    returns the buffer, the view and the host canary image."""
    host = canary(offset + a.size + GUARD, dtype)
    buf = to_dev(host, dtype)
    view = buf[offset:offset + a.size].view(a.shape)
    view.copy_(synth.to_torch(np.ascontiguousarray(a), dtype).to(DEV))
    return buf, view, host


def check_buffer(buf, host, offset, n, shape, want, dtype, what):
    got = synth.from_torch(buf)
    assert np.array_equal(got[:offset], host[:offset]), f"{what}: canary before x changed"
    assert np.array_equal(got[offset + n:], host[offset + n:]), f"{what}: canary after x changed"
    assert_same(got[offset:offset + n].reshape(shape), want, dtype, what)


@pytest.mark.parametrize("k", range(N_TABLE))
def test_fuzz_table(k):
    c = fc.table_case(k)
    x, g, r1p, r2p = fc.table_inputs(c)
    lo, L = c.r_offset, c.sl.L
    c1, s1 = to_dev(r1p, c.dtype)[..., lo:lo + L], to_dev(r2p, c.dtype)[..., lo:lo + L]
    r1, r2 = np.ascontiguousarray(r1p[..., lo:lo + L]), np.ascontiguousarray(r2p[..., lo:lo + L])
    for direction, inp in (("fwd", x), ("bwd", g)):
        buf, view, host = in_buffer(inp, c.x_offset, c.dtype)
        fn = binding.rope_partial_inplace_fwd_mode if direction == "fwd" else \
            binding.rope_partial_inplace_bwd_mode
        fn(view, c1, s1, c.sl.start, c.sl.end, c.mode)
        torch.cuda.synchronize()
        ofn = oracle.fwd if direction == "fwd" else oracle.bwd
        want = ofn(inp, r1, r2, c.dtype, c.sl.start, c.sl.end, oracle.GATHER_CHAIN, c.mode)
        check_buffer(buf, host, c.x_offset, inp.size, c.shape, want, c.dtype, f"{c} {direction}")


@pytest.mark.parametrize("k", range(N_HOST))
def test_fuzz_host_buffers(k):
    """The zero-copy calls on page-locked host tensors (interleave mode):
    x at an element offset inside a pinned canary buffer, cos/sin as views
    into padded pinned rows."""
    c = fc.table_case(k)
    x, g, r1p, r2p = fc.table_inputs(c)
    lo, L = c.r_offset, c.sl.L
    td = synth.TORCH_DTYPE[c.dtype]
    c1 = synth.to_torch(r1p, c.dtype).pin_memory()[..., lo:lo + L]
    s1 = synth.to_torch(r2p, c.dtype).pin_memory()[..., lo:lo + L]
    r1, r2 = np.ascontiguousarray(r1p[..., lo:lo + L]), np.ascontiguousarray(r2p[..., lo:lo + L])
    for direction, inp in (("fwd", x), ("bwd", g)):
        host = canary(c.x_offset + inp.size + GUARD, c.dtype)
        buf = synth.to_torch(host.copy(), c.dtype).pin_memory()
        assert buf.dtype == td
        view = buf[c.x_offset:c.x_offset + inp.size].view(inp.shape)
        view.copy_(synth.to_torch(np.ascontiguousarray(inp), c.dtype))
        fn = binding.rope_partial_inplace_fwd_host if direction == "fwd" else \
            binding.rope_partial_inplace_bwd_host
        fn(view, c1, s1, c.sl.start, c.sl.end)
        torch.cuda.synchronize()
        ofn = oracle.fwd if direction == "fwd" else oracle.bwd
        want = ofn(inp, r1, r2, c.dtype, c.sl.start, c.sl.end)
        check_buffer(buf, host, c.x_offset, inp.size, c.shape, want, c.dtype,
                     f"{c} host {direction}")


@pytest.mark.parametrize("k", range(N_QK))
def test_fuzz_qk(k):
    c = fc.qk_case(k)
    q, kk, r1, r2 = fc.qk_inputs(c)
    c1, s1 = to_dev(r1, c.dtype), to_dev(r2, c.dtype)
    qsl, ksl = c.q[2:], c.k[2:]
    for direction in ("fwd", "bwd"):
        qb, qv, qh = in_buffer(q, c.q_offset, c.dtype)
        kb, kv, kh = in_buffer(kk, c.k_offset, c.dtype)
        fn = binding.rope_partial_inplace_fwd_qk if direction == "fwd" else \
            binding.rope_partial_inplace_bwd_qk
        fn(qv, kv, c1, s1, qsl, ksl)
        torch.cuda.synchronize()
        d = oracle.FWD if direction == "fwd" else oracle.BWD
        wq, wk = oracle.rope_qk(d, q, kk, r1, r2, c.dtype, qsl, ksl)
        check_buffer(qb, qh, c.q_offset, q.size, q.shape, wq, c.dtype, f"{c} q {direction}")
        check_buffer(kb, kh, c.k_offset, kk.size, kk.shape, wk, c.dtype, f"{c} k {direction}")


@pytest.mark.parametrize("k", range(N_POS))
def test_fuzz_positions(k):
    c = fc.pos_case(k)
    x, p = fc.pos_inputs(c)
    pd = torch.from_numpy(p).to(DEV)
    for direction in ("fwd", "bwd"):
        xd = to_dev(x, c.dtype)
        fn = binding.rope_partial_inplace_fwd_pos if direction == "fwd" else \
            binding.rope_partial_inplace_bwd_pos
        fn(xd, pd, c.sl.start, c.sl.end, 10000.0, c.mode)
        torch.cuda.synchronize()
        d = oracle.FWD if direction == "fwd" else oracle.BWD
        want = oracle.rope_pos(d, x, p, 10000.0, c.dtype, c.sl.start, c.sl.end, c.mode)
        assert_close_pos(synth.from_torch(xd), want, oracle.widen(x, c.dtype), c.dtype,
                         c.sl.start, c.sl.end, c.mode, f"{c} {direction}")

"""GPU parity of the call that computes cos/sin from positions, against the
oracle's fp64-derived fp32 table.

The kernel's cos/sin are within 8e-7 of the exact values (angle formed and
reduced in fp32 with a three-part 2*pi, then the hardware sine/cosine on
[-pi, pi]), where the oracle uses the exact values rounded to fp32.  A
lane y = x_m c - x_n s (or its partner) then differs by at most
8e-7 * (|x_m| + |x_n|) before the final rounding, so the bar is that, with
margin: within 1e-6 * (|x_m| + |x_n|) plus the final rounding (2 ulp of
fp32, 1 ulp of bf16 / fp16).  In lanes where the two products cancel that
can be several units in the last place of y, so a pure ulp bound would be
wrong.  Every byte outside the slice is bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, assert_close_pos, to_dev
from place_partial_rope_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def run(direction, x, positions, dtype, start, end, mode, base=10000.0):
    xd = to_dev(x, dtype)
    pd = torch.from_numpy(np.ascontiguousarray(positions, dtype=np.int32)).to(DEV)
    fn = binding.rope_partial_inplace_fwd_pos if direction == "fwd" else binding.rope_partial_inplace_bwd_pos
    fn(xd, pd, start, end, base, mode)
    torch.cuda.synchronize()
    return synth.from_torch(xd)


def check(direction, x, positions, dtype, start, end, mode, what, base=10000.0):
    got = run(direction, x, positions, dtype, start, end, mode, base)
    d = oracle.FWD if direction == "fwd" else oracle.BWD
    want = oracle.rope_pos(d, x, positions, base, dtype, start, end, mode)
    assert_close_pos(got, want, oracle.widen(x, dtype), dtype, start, end, mode, what)


@pytest.mark.parametrize("mode", ["interleave", "half"])
@pytest.mark.parametrize("name", ["gqa", "mla_decode_q", "large_unaligned"])
def test_named_shapes_with_positions(name, mode):
    w = synth.WORKLOADS[name]
    x = synth.normal(w.shape, w.dtype, w.seed)
    pos = synth.positions(w)[..., 0].astype(np.int32)  # (Br, Sr) one position per (b, s)
    for direction in w.directions:
        inp = x if direction == "fwd" else synth.normal(w.shape, w.dtype, w.seed + 500)
        check(direction, inp, pos, w.dtype, w.start, w.end, mode, f"{name} {mode} {direction}")


SWEEP = [
    ((2, 5, 3, 64), 0, 64, (2, 5)),
    ((2, 5, 3, 64), 2, 58, (1, 5)),
    ((2, 5, 3, 64), 3, 61, (2, 1)),        # odd start
    ((3, 4, 7, 48), 1, 3, (1, 1)),         # one pair, one position for all
    ((1, 7, 5, 1024), 0, 1024, (1, 7)),    # the largest slice: 512 angles
    ((2, 3, 13, 24), 6, 22, (2, 3)),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("mode", ["interleave", "half"])
@pytest.mark.parametrize("k", range(len(SWEEP)))
def test_positions_sweep(dtype, mode, k):
    shape, st, en, pshape = SWEEP[k]
    x = synth.normal(shape, dtype, 400 + k)
    pos = np.random.default_rng(k).integers(0, 40000, size=pshape).astype(np.int32)
    for direction in ("fwd", "bwd"):
        check(direction, x, pos, dtype, st, en, mode, f"{shape} [{st},{en}) {direction}")


@pytest.mark.parametrize("mode", ["interleave", "half"])
def test_largest_exact_positions_and_other_bases(mode):
    """Positions up to 2^24 - 1 (the largest exact in fp32), and bases other
    than 10000."""
    x = synth.normal((2, 6, 4, 64), "fp32", 7)
    pos = np.array([[0, 1, 2**20, 2**23 + 3, 2**24 - 1, 12345],
                    [-5, -2**22, 99, 7, 2**24 - 2, 500000]], np.int32)
    for base in (10000.0, 500000.0, 2.0):
        for direction in ("fwd", "bwd"):
            check(direction, x, pos, "fp32", 0, 64, mode, f"base {base} {direction}", base)


def test_position_zero_is_the_identity_on_the_gpu():
    x = synth.normal((2, 3, 4, 32), "bf16", 3)
    got = run("fwd", x, np.zeros((1, 1), np.int32), "bf16", 0, 32, "interleave")
    assert np.array_equal(got, x)


@pytest.mark.parametrize("mode", ["interleave", "half"])
@pytest.mark.parametrize("base,L", [(10000.0, 64), (10000.0, 2), (500000.0, 128), (1e6, 512),
                                    (2.0, 16)])
def test_kernel_cos_sin_error_bound(base, L, mode):
    """The premise of the bar above, measured: with unit pairs (x_m, x_n) =
    (1, 0) the forward writes the kernel's own cos and sin (1*c - 0*s = c and
    0*c + 1*s = s, each product and sum exact), so comparing them with the
    fp64 cos/sin of p * base^(-2k/L) gives the kernel's angle error directly.
    Positions span [-2^24, 2^24), where they are exact in fp32, with the
    ends and small values included.  ("ANE实战 RoPE位置编码在MIL中的纯ANE实现",
    sections 先搞懂RoPE and 第一步: theta_k = p / base^(2k/L).)"""
    rng = np.random.default_rng(2024)
    ends = np.array([0, 1, -1, 2, 3, 7, 1000, -1000, 2**23, -2**23, 2**24 - 1, -2**24,
                     2**24 - 2, 12345678, -9876543], np.int64)
    p = np.concatenate([ends, rng.integers(-2**24, 2**24, size=4096 - ends.size)]).astype(np.int32)
    S = p.size
    x = np.zeros((1, S, 1, L), np.float32)
    if mode == "half":
        x[..., :L // 2] = 1.0   # x_m = 1 in the first half, x_n = 0 in the second
    else:
        x[..., 0::2] = 1.0      # x_m = 1 in even lanes, x_n = 0 in odd lanes
    got = run("fwd", x, p[None, :], "fp32", 0, L, mode, base).astype(np.float64)
    k = np.arange(L // 2, dtype=np.float64)
    theta = p.astype(np.float64)[:, None] * np.array([math.pow(base, -2.0 * kk / L) for kk in k])
    if mode == "half":
        c, s = got[0, :, 0, :L // 2], got[0, :, 0, L // 2:]
    else:
        c, s = got[0, :, 0, 0::2], got[0, :, 0, 1::2]
    err = max(np.abs(c - np.cos(theta)).max(), np.abs(s - np.sin(theta)).max())
    print(f"base {base} L {L} {mode}: max |cos/sin error| {err:.3e}")
    assert err <= 8e-7, err

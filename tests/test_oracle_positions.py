"""Pins for the oracle of the call that computes cos/sin from positions.

The angle of pair k at position p is theta_k = p / 10000^(2k/L) ("ANE实战
RoPE位置编码在MIL中的纯ANE实现", section 先搞懂RoPE: theta = p / 10000^(2i/h);
section 第一步: the table over positions and pairs).  These checks pin that
recipe without retyping it: the angle read back from a rotated unit vector
against an independent evaluation with math.exp/math.log, the group law of
rotations, RoPE's relative-position property from the same section (the
query-key product depends only on the position difference), the identity at
position 0, and agreement with the input generator's table.
"""
import math

import numpy as np
import pytest

import oracle
from place_partial_rope_gb300 import synth

MODES = ("interleave", "half")


def first(a, mode):
    return a[..., 0::2] if mode == "interleave" else a[..., : a.shape[-1] // 2]


def second(a, mode):
    return a[..., 1::2] if mode == "interleave" else a[..., a.shape[-1] // 2:]


@pytest.mark.parametrize("mode", MODES)
def test_angle_of_each_pair(mode):
    """Rotate the unit vector (1, 0) of every pair (fp32, so the result is
    (cos, sin) of the fp32 table) and read its angle back with atan2."""
    L, base = 16, 10000.0
    positions = np.array([[0, 1, 7, 100, 4095, 30000]], np.int32)
    S = positions.shape[1]
    x = np.zeros((1, S, 1, L), np.float32)
    if mode == "interleave":
        x[..., 0::2] = 1.0
    else:
        x[..., : L // 2] = 1.0
    y = oracle.rope_pos(oracle.FWD, x, positions, base, "fp32", 0, L, mode)
    got = np.arctan2(second(y, mode).astype(np.float64), first(y, mode).astype(np.float64))[0, :, 0]
    for si in range(S):
        p = int(positions[0, si])
        for k in range(L // 2):
            omega = math.exp(-(2.0 * k / L) * math.log(base))
            want = math.remainder(p * omega, 2.0 * math.pi)
            err = abs(math.remainder(float(got[si, k]) - want, 2.0 * math.pi))
            assert err < 2e-6, (p, k, got[si, k], want)


@pytest.mark.parametrize("mode", MODES)
def test_rotations_compose(mode):
    """R(p1) then R(p2) equals R(p1 + p2), within fp32 rounding."""
    L, base = 32, 10000.0
    x = synth.normal((2, 5, 3, 40), "fp32", 3)
    p1 = np.array([[3, 10, 0, 77, 500]], np.int32)
    p2 = np.array([[4, 1, 9, 23, 1000]], np.int32)
    a = oracle.rope_pos(oracle.FWD, oracle.rope_pos(oracle.FWD, x, p1, base, "fp32", 4, 36, mode),
                        p2, base, "fp32", 4, 36, mode)
    b = oracle.rope_pos(oracle.FWD, x, p1 + p2, base, "fp32", 4, 36, mode)
    norm = np.sqrt(first(x[..., 4:36], mode).astype(np.float64) ** 2 +
                   second(x[..., 4:36], mode).astype(np.float64) ** 2)
    diff = np.abs(a[..., 4:36].astype(np.float64) - b[..., 4:36])
    assert (np.maximum(first(diff, mode), second(diff, mode)) / norm).max() < 2e-6
    assert np.array_equal(a[..., :4], x[..., :4]) and np.array_equal(a[..., 36:], x[..., 36:])


@pytest.mark.parametrize("mode", MODES)
def test_relative_position_property(mode):
    """<rope(q, m), rope(k, n)> over the slice depends only on m - n."""
    L, base = 64, 10000.0
    q = synth.normal((1, 1, 1, L), "fp32", 11)
    k = synth.normal((1, 1, 1, L), "fp32", 12)

    def dot(m, n):
        qm = oracle.rope_pos(oracle.FWD, q, np.array([[m]], np.int32), base, "fp32", 0, L, mode)
        kn = oracle.rope_pos(oracle.FWD, k, np.array([[n]], np.int32), base, "fp32", 0, L, mode)
        return float(np.sum(qm.astype(np.float64) * kn))

    for delta in (0, 1, 5, 300):
        vals = [dot(m + delta, m) for m in (0, 17, 1000, 20000)]
        scale = float(np.sum(np.abs(q.astype(np.float64)) * 1) * np.abs(k).max())
        assert max(vals) - min(vals) <= 1e-5 * scale, (delta, vals)
    assert abs(dot(0, 0) - float(np.sum(q.astype(np.float64) * k))) < 1e-5


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
@pytest.mark.parametrize("mode", MODES)
def test_position_zero_is_the_identity(dtype, mode):
    x = synth.normal((2, 3, 4, 24), dtype, 5)
    pos = np.zeros((2, 3), np.int32)
    for d in (oracle.FWD, oracle.BWD):
        y = oracle.rope_pos(d, x, pos, 10000.0, dtype, 4, 20, mode)
        assert np.array_equal(y.view(np.uint8), x.view(np.uint8))


@pytest.mark.parametrize("mode", MODES)
def test_table_agrees_with_the_input_recipe(mode):
    """The oracle's fp32 table equals the input generator's fp32 table (two
    separately written statements of the same recipe)."""
    pos = np.array([[0, 3, 999, 32767]], np.int64)
    c, s = oracle.position_table(pos, 64, 10000.0, mode)
    rc, rs = synth.rope_table(pos[..., None], 64, "fp32", layout=mode)
    assert np.array_equal(c, rc) and np.array_equal(s, rs)


def test_positions_equal_the_table_call_in_fp32():
    """In fp32 the positions call is the table call with that table."""
    x = synth.normal((2, 4, 3, 32), "fp32", 9)
    pos = np.array([[5, 6, 7, 8], [100, 101, 102, 103]], np.int32)
    c, s = oracle.position_table(pos, 24, 10000.0)
    a = oracle.rope_pos(oracle.BWD, x, pos, 10000.0, "fp32", 4, 28)
    b = oracle.bwd(x, c, s, "fp32", 4, 28)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))

"""Pins for the oracle's IEEE 754 storage conversions.

The oracle rounds binary32 to bfloat16 and binary16 with its own code (round
to nearest, ties to even: the CAST_RINT write-back of "CANN ops-transformer
inplace_partial_rotary_mul", section "Tiling 与 Kernel 的工程细节").  Here that
code is checked against library conversions that implement the same IEEE
rule: numpy's float32 -> float16 and torch's CPU float32 -> bfloat16, over
every exact tie, the neighbours of every tie, and a dense stride of all 2^32
binary32 bit patterns.  The widening conversions are checked exhaustively.
"""
import numpy as np
import pytest
import torch

import oracle


def _all_strided_f32(step=4099):
    bits = np.arange(0, 2**32, step, dtype=np.uint64).astype(np.uint32)
    return bits.view(np.float32)


def _ties_and_neighbours(low_bits_of_half: int):
    """For every possible kept-part pattern: the exact tie and +-1 ulp of it."""
    hi = np.arange(0, 2**16, dtype=np.uint32) << 16
    out = []
    for kept_shift in (low_bits_of_half,):
        half = np.uint32(1 << (kept_shift - 1))
        for delta in (-1, 0, 1):
            out.append(hi | np.uint32(int(half) + delta))
    return np.concatenate(out).view(np.float32)


def _assert_same_or_both_nan(got_bits, ref_bits, widen):
    got_f = widen(got_bits)
    ref_f = widen(ref_bits)
    nan = np.isnan(ref_f)
    assert np.array_equal(np.isnan(got_f), nan)
    bad = np.nonzero(got_bits[~nan] != ref_bits[~nan])[0]
    assert bad.size == 0, f"{bad.size} mismatches, first at index {bad[:5]}"


def _torch_bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_f32_to_bf16_matches_torch_dense_and_ties():
    vals = np.concatenate([_all_strided_f32(), _ties_and_neighbours(16)])
    got = oracle.f32_to_bf16(vals)
    ref = _torch_bf16_bits(vals)
    _assert_same_or_both_nan(got, ref, oracle.bf16_to_f32)


def test_f32_to_f16_matches_numpy_dense():
    vals = _all_strided_f32()
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16(vals)
    _assert_same_or_both_nan(got, ref, oracle.f16_to_f32)


def test_f32_to_f16_matches_numpy_at_every_tie():
    # the binary32 midpoints between consecutive binary16 values, including
    # the subnormal range and the overflow threshold, and +-1 binary32 ulp
    h = np.arange(0, 0x7C00, dtype=np.uint16)  # all finite non-negative halves
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)  # exact: midpoint needs <= 12 bits
    mid_bits = mid.view(np.uint32)
    cand = np.concatenate([mid_bits - 1, mid_bits, mid_bits + 1]).view(np.float32)
    cand = np.concatenate([cand, -cand])
    with np.errstate(over="ignore"):
        ref = cand.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16(cand)
    _assert_same_or_both_nan(got, ref, oracle.f16_to_f32)


def test_specials():
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 65504.0, 65519.99, 65520.0,
                         2.0**-24, 2.0**-25, 2.0**-25 * 1.0000001, 2.0**-149, 3.4e38],
                        dtype=np.float32)
    with np.errstate(over="ignore"):
        ref16 = specials.astype(np.float16).view(np.uint16)
    _assert_same_or_both_nan(oracle.f32_to_f16(specials), ref16, oracle.f16_to_f32)
    _assert_same_or_both_nan(oracle.f32_to_bf16(specials), _torch_bf16_bits(specials),
                             oracle.bf16_to_f32)
    # signed zero survives both directions
    assert oracle.f32_to_f16(np.array([-0.0], np.float32))[0] == 0x8000
    assert oracle.f32_to_bf16(np.array([-0.0], np.float32))[0] == 0x8000


@pytest.mark.parametrize("kind", ["fp16", "bf16"])
def test_widening_exhaustive(kind):
    h = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    if kind == "fp16":
        got = oracle.f16_to_f32(h)
        ref = h.view(np.float16).astype(np.float32)
    else:
        got = oracle.bf16_to_f32(h)
        ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))

"""Helpers for the GPU parity tests: run the CUDA path through the C ABI
binding on host arrays, and compare results with the oracle's."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from place_partial_rope_gb300 import binding, synth

DEV = torch.device("cuda:0")


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    return synth.to_torch(np.ascontiguousarray(a), dtype).to(DEV)


def run_cuda(direction: str, x, r1, r2, dtype, start, end, stream=None) -> np.ndarray:
    """Copy to the GPU, run the forward or backward in place, copy back."""
    xd, c, s = to_dev(x, dtype), to_dev(r1, dtype), to_dev(r2, dtype)
    fn = binding.rope_partial_inplace_fwd if direction == "fwd" else binding.rope_partial_inplace_bwd
    fn(xd, c, s, start, end, stream=stream)
    torch.cuda.synchronize()
    return synth.from_torch(xd)


def run_oracle(direction: str, x, r1, r2, dtype, start, end) -> np.ndarray:
    fn = oracle.fwd if direction == "fwd" else oracle.bwd
    return fn(x, r1, r2, dtype, start, end)


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


def assert_same(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    """Bit-exact, except that two NaNs match whatever their payloads."""
    assert got.shape == want.shape, (got.shape, want.shape)
    gb, wb = bits(np.ascontiguousarray(got)).ravel(), bits(np.ascontiguousarray(want)).ravel()
    diff = np.nonzero(gb != wb)[0]
    if diff.size == 0:
        return
    gv = oracle.widen(got.ravel()[diff], dtype)
    wv = oracle.widen(want.ravel()[diff], dtype)
    real = diff[~(np.isnan(gv) & np.isnan(wv))]
    assert real.size == 0, (
        f"{what}: {real.size} of {gb.size} lanes differ; first flat indices {real[:6]}, "
        f"got {oracle.widen(got.ravel()[real[:6]], dtype)} "
        f"want {oracle.widen(want.ravel()[real[:6]], dtype)}")


def split(a, mode):
    if mode == "interleave":
        return a[..., 0::2], a[..., 1::2]
    h = a.shape[-1] // 2
    return a[..., :h], a[..., h:]


def storage_ulp(bits: np.ndarray, dtype: str) -> np.ndarray:
    """The spacing of the storage type at each value (from its bit pattern)."""
    if dtype == "fp32":
        return np.spacing(np.abs(bits.view(np.float32))).astype(np.float64)
    mag = (bits & 0x7FFF).astype(np.uint16)
    nxt = np.minimum(mag + 1, 0x7BFF if dtype == "fp16" else 0x7F7F).astype(np.uint16)
    return np.abs(oracle.widen(nxt, dtype).astype(np.float64) - oracle.widen(mag, dtype))


def assert_close_pos(got, want, x, dtype, start, end, mode, what):
    """The bar for the call that computes cos/sin from positions: lanes
    within 1e-6 * (|x_m| + |x_n|) plus the final rounding of the oracle's
    fp32-table result; every byte outside the slice bit-exact; and for
    16-bit types, fewer than 2 % of the lanes off by their final rounding."""
    assert np.array_equal(got[..., :start].view(np.uint8), want[..., :start].view(np.uint8)), what
    assert np.array_equal(got[..., end:].view(np.uint8), want[..., end:].view(np.uint8)), what
    g, w = got[..., start:end], want[..., start:end]
    xs = x[..., start:end].astype(np.float64)
    xm, xn = split(xs, mode)
    mag = np.abs(xm) + np.abs(xn)
    mag = np.concatenate([mag, mag], axis=-1) if mode == "half" else np.repeat(mag, 2, axis=-1)
    rounding = (2 if dtype == "fp32" else 1) * storage_ulp(np.ascontiguousarray(w), dtype)
    tol = 1e-6 * mag + rounding
    err = np.abs(oracle.widen(np.ascontiguousarray(g), dtype).astype(np.float64) -
                 oracle.widen(np.ascontiguousarray(w), dtype))
    assert np.all(err <= tol), f"{what}: max err {err.max()}, worst ratio {(err / tol).max()}"
    if dtype != "fp32" and err.size >= 2000:  # a rate: only meaningful over many lanes
        assert (err > 0).mean() < 0.02, f"{what}: {(err > 0).mean():.3%} of lanes differ"

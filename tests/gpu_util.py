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

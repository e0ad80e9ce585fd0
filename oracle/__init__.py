"""CPU oracle for the in-place partial interleaved rotary embedding.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  It shares no code with the CUDA path, and the CUDA path
never imports it.

Contents
--------
* ``rope_oracle.c`` -- the scalar C statement of the forward and backward
  (gather-chain and pair-rotation formulations) and the IEEE 754 storage
  conversions, built into ``librope_oracle.so`` by :func:`build`.
* ``rope_mil.py`` -- a third, array-level formulation (reshape / slice /
  negate / concat), written with numpy float32 operations.

Two rotary modes: "interleave" (the page's mode, pairs (2i, 2i+1)) and
"half" (the half-split rotate_half mode, pairs (i, i + L/2)).

Sources: "CANN ops-transformer inplace_partial_rotary_mul" (formula section
and its kernel op chain; tiling section for FP32 compute with CAST_RINT);
"ANE实战 RoPE位置编码在MIL中的纯ANE实现" (rotate_half lowering table, backward
section).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, special cases, invariants, brute-force Jacobians, library
conversions and a hand-worked example); none is "parity unpinned".
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rope_oracle.c")
LIB = os.path.join(HERE, "librope_oracle.so")

BF16, FP16, FP32 = 0, 1, 2
DTYPE_CODES = {"bf16": BF16, "fp16": FP16, "fp32": FP32}
GATHER_CHAIN, PAIR_ROTATION = 0, 1
FWD, BWD = 0, 1
INTERLEAVE, HALF = 1, 2
MODE_CODES = {"interleave": INTERLEAVE, "half": HALF}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", LIB, SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return LIB


def _open(path):
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_rope.restype = ctypes.c_int
    lib.oracle_rope.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                i64p, i64p, i64p, i64p, ctypes.c_int64, ctypes.c_int64]
    lib.oracle_rope_mixed.restype = ctypes.c_int
    lib.oracle_rope_mixed.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p] * 3 + \
        [ctypes.c_int64] * 4 + [i64p] * 4 + [ctypes.c_int64] * 2
    for name in ("oracle_f32_to_bf16_n", "oracle_f32_to_f16_n",
                 "oracle_bf16_to_f32_n", "oracle_f16_to_f32_n"):
        fn = getattr(lib, name)
        fn.restype = None
        fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _open(LIB)
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily route every oracle call through another build of the
    oracle source (the mutation tests use this to run the pins against
    deliberately broken copies)."""
    global _lib
    saved = _load()
    _lib = _open(path)
    try:
        yield
    finally:
        _lib = saved


def _i64x4(vals):
    return (ctypes.c_int64 * 4)(*[int(v) for v in vals])


def _elem_strides(arr: np.ndarray):
    return [s // arr.itemsize for s in arr.strides]


def rope(direction: int, x: np.ndarray, r1: np.ndarray, r2: np.ndarray, dtype: str,
         start: int, end: int, formulation: int = GATHER_CHAIN,
         mode: str = "interleave") -> np.ndarray:
    """Return a copy of ``x`` with the forward (``FWD``) or backward (``BWD``)
    applied to lanes ``[start, end)`` of its last axis, pairing lanes
    (2i, 2i+1) (``mode="interleave"``) or (i, i + L/2) (``mode="half"``).

    ``x`` is a contiguous 4-D array (B, S, N, D) holding the storage type:
    float32 for ``fp32``, uint16 bit patterns for ``bf16`` and ``fp16``.
    ``r1`` (cos) and ``r2`` (sin) are 4-D arrays of the same storage type that
    broadcast against the slice; they may be strided views (numpy strides in
    bytes are converted to element strides).
    """
    lib = _load()
    code = DTYPE_CODES[dtype]
    want = np.float32 if code == FP32 else np.uint16
    for a in (x, r1, r2):
        if a.dtype != want or a.ndim != 4:
            raise ValueError(f"oracle expects 4-D {want} arrays for {dtype}")
    out = np.ascontiguousarray(x).copy()
    B, S, N, D = out.shape
    rc = lib.oracle_rope(direction, formulation, MODE_CODES[mode], code,
                         out.ctypes.data, r1.ctypes.data, r2.ctypes.data, B, S, N, D,
                         _i64x4(r1.shape), _i64x4(_elem_strides(r1)),
                         _i64x4(r2.shape), _i64x4(_elem_strides(r2)), start, end)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def fwd(x, r1, r2, dtype, start, end, formulation=GATHER_CHAIN, mode="interleave"):
    return rope(FWD, x, r1, r2, dtype, start, end, formulation, mode)


def bwd(g, r1, r2, dtype, start, end, formulation=GATHER_CHAIN, mode="interleave"):
    return rope(BWD, g, r1, r2, dtype, start, end, formulation, mode)


def position_table(positions: np.ndarray, L: int, base: float, mode: str = "interleave"):
    """cos/sin of every position, for the call that computes them in the
    kernel: theta_k = p / base^(2k/L) for pair k in [0, L/2) ("ANE实战
    RoPE位置编码在MIL中的纯ANE实现", sections 先搞懂RoPE and 第一步), computed in
    float64 and rounded once to float32.  Pair k's value fills lanes 2k and
    2k+1 (interleave) or k and k + L/2 (half).  Returns float32 arrays of
    shape positions.shape + (1, L), i.e. (Bp, Sp, 1, L)."""
    k = np.arange(L // 2, dtype=np.float64)
    omega = np.power(float(base), -2.0 * k / L)
    theta = positions.astype(np.float64)[..., None] * omega
    c, s = np.cos(theta), np.sin(theta)
    if mode == "half":
        c, s = np.concatenate([c, c], axis=-1), np.concatenate([s, s], axis=-1)
    else:
        c, s = np.repeat(c, 2, axis=-1), np.repeat(s, 2, axis=-1)
    c = np.ascontiguousarray(c.astype(np.float32)[..., None, :])
    s = np.ascontiguousarray(s.astype(np.float32)[..., None, :])
    return c, s


def rope_pos(direction: int, x: np.ndarray, positions: np.ndarray, base: float, dtype: str,
             start: int, end: int, mode: str = "interleave",
             formulation: int = GATHER_CHAIN) -> np.ndarray:
    """The operation with cos/sin computed from positions (one int32 per
    (b, s), shape (Bp, Sp) broadcasting against (B, S)): the table of
    position_table() -- float32 values, not rounded to x's type -- then the
    same op chain as rope()."""
    lib = _load()
    code = DTYPE_CODES[dtype]
    want = np.float32 if code == FP32 else np.uint16
    if x.dtype != want or x.ndim != 4:
        raise ValueError(f"oracle expects a 4-D {want} array for {dtype}")
    c, s = position_table(np.asarray(positions), end - start, base, mode)
    out = np.ascontiguousarray(x).copy()
    B, S, N, D = out.shape
    rc = lib.oracle_rope_mixed(direction, formulation, MODE_CODES[mode], code, FP32,
                               out.ctypes.data, c.ctypes.data, s.ctypes.data, B, S, N, D,
                               _i64x4(c.shape), _i64x4(_elem_strides(c)),
                               _i64x4(s.shape), _i64x4(_elem_strides(s)), start, end)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def rope_qk(direction: int, q: np.ndarray, k: np.ndarray, r1: np.ndarray, r2: np.ndarray,
            dtype: str, q_slice, k_slice, formulation: int = GATHER_CHAIN):
    """The fused query + key call by its definition: the operation applied to
    q and to k with the same cos/sin rows (the RoPE stage of
    "ascend-transformer-boost MlaPreprocessOperation", section 3: rotate
    Q[..., :qRopeDim] and K[..., :kRopeDim] with cos/sin passed in).  Pinned
    through the single-tensor pins, since it is nothing but two of them."""
    return (rope(direction, q, r1, r2, dtype, q_slice[0], q_slice[1], formulation),
            rope(direction, k, r1, r2, dtype, k_slice[0], k_slice[1], formulation))


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_f32_to_bf16_n(a.ctypes.data, out.ctypes.data, a.size)
    return out


def f32_to_f16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_f32_to_f16_n(a.ctypes.data, out.ctypes.data, a.size)
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().oracle_bf16_to_f32_n(h.ctypes.data, out.ctypes.data, h.size)
    return out


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().oracle_f16_to_f32_n(h.ctypes.data, out.ctypes.data, h.size)
    return out


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array -> float32 values, through the oracle's own conversions."""
    if dtype == "fp32":
        return np.asarray(a, np.float32)
    return bf16_to_f32(a) if dtype == "bf16" else f16_to_f32(a)


def narrow(a: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> storage array, through the oracle's own RNE rounding."""
    if dtype == "fp32":
        return np.asarray(a, np.float32)
    return f32_to_bf16(a) if dtype == "bf16" else f32_to_f16(a)

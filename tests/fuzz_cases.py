"""Seeded random cases for the fuzz tests: shapes, slices, broadcast forms,
buffer offsets and padded cos/sin rows, drawn on the host.  Nothing here
computes the operation; the oracle and the CUDA path both take these draws
as plain inputs.

The slice rules are those of "CANN ops-transformer inplace_partial_rotary_mul",
section 约束说明: D even and at most 1024, 0 <= start <= end <= D, end - start
even, any start (odd starts included), cos/sin broadcast against
(B, S, N, end - start).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from place_partial_rope_gb300 import synth

SEED = 20261202
HEAD_DIMS = (2, 4, 6, 8, 10, 12, 16, 20, 24, 30, 32, 40, 48, 64, 66, 96, 128, 130, 160, 192,
             256, 512, 1024)
MAX_ELEMS = 48_000          # per tensor: keeps every case to milliseconds
QK_FORMS = ("BS1D", "1S1D", "B11D", "111D")   # one cos/sin row per (batch, position)


@dataclass
class Slice:
    D: int
    start: int
    end: int

    @property
    def L(self) -> int:
        return self.end - self.start


@dataclass
class TableCase:
    dtype: str
    mode: str
    shape: tuple
    sl: Slice
    form: str
    x_offset: int      # elements between the buffer's start and x
    r_offset: int      # elements between a padded cos/sin row's start and the slice
    r_pad: int         # padded row length minus L
    seed: int


@dataclass
class QKCase:
    dtype: str
    bs: tuple
    q: tuple           # (Nq, Dq, start, end)
    k: tuple           # (Nk, Dk, start, end)
    form: str
    q_offset: int
    k_offset: int
    seed: int


@dataclass
class PosCase:
    dtype: str
    mode: str
    shape: tuple
    sl: Slice
    pos_shape: tuple
    seed: int


def _rng(kind: int, k: int) -> np.random.Generator:
    return np.random.default_rng([SEED, kind, k])


def _slice(rng, D: int, L: int | None = None, aligned: bool = False) -> Slice:
    """An even-length slice of a row of D: full, a power-of-two number of
    pairs, any even length, or empty; its start odd a third of the time
    when there is room (a multiple of 8 when `aligned`)."""
    if L is None:
        u = rng.random()
        if u < 0.05:
            L = 0
        elif u < 0.3:
            L = D
        elif u < 0.55:
            L = 2 * int(2 ** rng.integers(0, int(np.log2(D // 2)) + 1))
        else:
            L = 2 * int(rng.integers(1, D // 2 + 1))
    room = D - L
    if room == 0:
        return Slice(D, 0, D)
    u = 0.5 if aligned else rng.random()
    if u < 0.35:
        start = 2 * int(rng.integers(0, (room + 1) // 2)) + 1 if room >= 1 else 0
    elif u < 0.6:
        start = 8 * int(rng.integers(0, room // 8 + 1))
    else:
        start = int(rng.integers(0, room + 1))
    start = min(start, room)
    return Slice(D, start, start + L)


def _bsn(rng, D: int, max_elems: int = MAX_ELEMS) -> tuple:
    rows = max(1, max_elems // D)
    N = int(rng.integers(1, min(20, rows) + 1))
    B = int(rng.integers(1, min(4, max(1, rows // N)) + 1))
    S = int(rng.integers(1, min(64, max(1, rows // (N * B))) + 1))
    return B, S, N


def table_case(k: int) -> TableCase:
    rng = _rng(1, k)
    dtype = synth.DTYPES[int(rng.integers(0, 3))]
    mode = "half" if rng.random() < 0.4 else "interleave"
    D = int(rng.choice(HEAD_DIMS))
    # two cases in five keep every pointer and stride 16-byte aligned, so
    # that the widest accesses are drawn too
    aligned = rng.random() < 0.4
    sl = _slice(rng, D, aligned=aligned)
    odd_words = not aligned and rng.random() < 0.25
    if odd_words:
        # an odd start with x and the cos/sin rows aligned to 4 bytes or more
        # (the odd-start kernel's lane per aligned vector of x): half the
        # slices a power-of-two number of pairs up to 32, half any length
        D = int(rng.choice([d for d in HEAD_DIMS if d >= 4]))
        if rng.random() < 0.5:
            L = 2 * int(2 ** rng.integers(0, min(5, int(np.log2((D - 2) // 2))) + 1))
        else:
            L = 2 * int(rng.integers(1, (D - 2) // 2 + 1))
        start = 2 * int(rng.integers(0, (D - L) // 2)) + 1
        sl = Slice(D, start, start + L)
    B, S, N = _bsn(rng, D)
    form = list(synth.BROADCAST_FORMS)[int(rng.integers(0, len(synth.BROADCAST_FORMS)))]
    if aligned:
        x_offset, r_offset, r_pad = 0, 0, int(rng.choice([0, 0, 8, 16]))
    elif odd_words:
        x_offset, r_offset = 2 * int(rng.integers(0, 5)), 2 * int(rng.integers(0, 2))
        r_pad = r_offset + 2 * int(rng.integers(0, 3))
    else:
        x_offset, r_offset = int(rng.integers(0, 5)), int(rng.integers(0, 4))
        r_pad = r_offset + int(rng.integers(0, 6))
    return TableCase(dtype, mode, (B, S, N, D), sl, form, x_offset, r_offset, r_pad, 5000 + k)


def qk_case(k: int) -> QKCase:
    rng = _rng(2, k)
    dtype = synth.DTYPES[int(rng.integers(0, 3))]
    Dq = int(rng.choice(HEAD_DIMS))
    Dk = int(rng.choice([d for d in HEAD_DIMS if d <= 256]))
    qs = _slice(rng, Dq)
    L = min(qs.L, Dk - Dk % 2)
    qs = _slice(rng, Dq, L)
    ks = _slice(rng, Dk, L)
    B, S, Nq = _bsn(rng, max(Dq, Dk), MAX_ELEMS // 2)
    Nk = int(rng.integers(0, 5))
    form = QK_FORMS[int(rng.integers(0, len(QK_FORMS)))]
    return QKCase(dtype, (B, S), (Nq, Dq, qs.start, qs.end), (Nk, Dk, ks.start, ks.end), form,
                  int(rng.integers(0, 5)), int(rng.integers(0, 5)), 7000 + k)


def pos_case(k: int) -> PosCase:
    rng = _rng(3, k)
    dtype = synth.DTYPES[int(rng.integers(0, 3))]
    mode = "half" if rng.random() < 0.4 else "interleave"
    D = int(rng.choice(HEAD_DIMS))
    sl = _slice(rng, D)
    B, S, N = _bsn(rng, D)
    pos_shape = (B if rng.random() < 0.5 else 1, S if rng.random() < 0.8 else 1)
    return PosCase(dtype, mode, (B, S, N, D), sl, pos_shape, 9000 + k)


def table_inputs(c: TableCase):
    """x, grad, and the padded cos/sin tensors (the slice is
    [r_offset, r_offset + L) of their last axis)."""
    x = synth.normal(c.shape, c.dtype, c.seed)
    g = synth.normal(c.shape, c.dtype, c.seed + 500)
    rs = synth.r_shape_for(c.form, c.shape, c.sl.L)
    r1, r2 = synth.random_table(rs[:3] + (c.sl.L + c.r_pad,), c.dtype, c.seed + 77)
    return x, g, r1, r2


def qk_inputs(c: QKCase):
    (B, S), (Nq, Dq, qs, qe), (Nk, Dk, _, _) = c.bs, c.q, c.k
    q = synth.normal((B, S, Nq, Dq), c.dtype, c.seed)
    kk = synth.normal((B, S, Nk, Dk), c.dtype, c.seed + 1)
    rs = synth.r_shape_for(c.form, (B, S, 1, Dq), qe - qs)
    r1, r2 = synth.random_table(rs, c.dtype, c.seed + 77)
    return q, kk, r1, r2


def pos_inputs(c: PosCase):
    x = synth.normal(c.shape, c.dtype, c.seed)
    p = _rng(4, c.seed).integers(-50_000, 50_000, size=c.pos_shape).astype(np.int32)
    return x, p

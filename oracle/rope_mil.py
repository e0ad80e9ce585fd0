"""Array-level formulation of the interleaved rotation (oracle formulation C).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.

It follows the operator decomposition printed for the rotate_half lowering
in "ANE实战 RoPE位置编码在MIL中的纯ANE实现" (section 第二步, the five-step
table): reshape the last axis into (pairs, 2); slice out the even lanes q_e
and the odd lanes q_o; multiply q_o by -1; concatenate (-q_o, q_e) on the
new axis and reshape back to the interleaved layout; then mul, mul, add with
the cos and sin tensors.  It applies to the slice of "CANN ops-transformer
inplace_partial_rotary_mul" (section 功能与计算公式): only lanes
[start, end) of the last axis change.

Arithmetic: numpy float32 elementwise multiply and add, each one IEEE
binary32 rounding (numpy never fuses them).  The storage conversions go
through the C oracle's IEEE routines (``oracle.widen`` / ``oracle.narrow``).

The backward here is the transposed rotation on the pairs
(dx_e = g_e c_e + g_o s_o, dx_o = g_o c_o - g_e s_e), with the same
decomposition: reshape, slice, multiply, negate, interleave, add.

Half-split mode (``mode="half"``) follows the page's prose definition of
rotate_half ("swap the two halves of the vector and negate the front
half"): x1, x2 = the halves, rotated = concat(-x2, x1).
"""
from __future__ import annotations

import numpy as np

from . import narrow, widen


def _pairs(a: np.ndarray) -> np.ndarray:
    return a.reshape(a.shape[:-1] + (a.shape[-1] // 2, 2))


def _interleave(even: np.ndarray, odd: np.ndarray) -> np.ndarray:
    both = np.concatenate([even[..., None], odd[..., None]], axis=-1)
    return both.reshape(both.shape[:-2] + (both.shape[-2] * 2,))


def _halves(a: np.ndarray):
    h = a.shape[-1] // 2
    return a[..., :h], a[..., h:]


def fwd(x, r1, r2, dtype, start, end, mode="interleave"):
    """Forward through reshape / slice / negate / concat, mul, mul, add."""
    out = np.array(x, copy=True)
    if end == start or out.size == 0:
        return out
    xs = widen(out[..., start:end], dtype)
    c = np.broadcast_to(widen(r1, dtype), xs.shape)
    s = np.broadcast_to(widen(r2, dtype), xs.shape)
    if mode == "half":
        x1, x2 = _halves(xs)
        q_rot = np.concatenate([x2 * np.float32(-1.0), x1], axis=-1)
    else:
        q = _pairs(xs)
        q_e, q_o = q[..., 0], q[..., 1]
        nq = q_o * np.float32(-1.0)
        q_rot = _interleave(nq, q_e)
    y = xs * c + q_rot * s
    out[..., start:end] = narrow(y, dtype)
    return out


def bwd(g, r1, r2, dtype, start, end, mode="interleave"):
    """Backward: the transposed rotation of the gradient, in the same style."""
    out = np.array(g, copy=True)
    if end == start or out.size == 0:
        return out
    gs = widen(out[..., start:end], dtype)
    c = np.broadcast_to(widen(r1, dtype), gs.shape)
    s = np.broadcast_to(widen(r2, dtype), gs.shape)
    t1 = gs * c
    if mode == "half":
        u1, u2 = _halves(gs * s)
        w = np.concatenate([u2, u1 * np.float32(-1.0)], axis=-1)
    else:
        u = _pairs(gs * s)
        u_e, u_o = u[..., 0], u[..., 1]
        w = _interleave(u_o, u_e * np.float32(-1.0))
    out[..., start:end] = narrow(t1 + w, dtype)
    return out

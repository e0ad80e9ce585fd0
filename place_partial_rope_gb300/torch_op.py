"""PyTorch operator and autograd for the in-place partial rotary embedding.

The user-facing API described by "CANN ops-transformer
inplace_partial_rotary_mul" (sections 函数原型与参数说明, 自动微分说明 and
图模式调用), on top of the C ABI:

    inplace_partial_rotary_mul(x, r1, r2, *, rotary_mode="interleave",
                               partial_slice=None) -> None

* Operator schema (namespace ``place_partial_rope``):
  ``inplace_partial_rotary_mul(Tensor(a!) x, Tensor r1, Tensor r2, *,
  str rotary_mode='interleave', int[2] partial_slice=[0, 0]) -> ()`` and
  ``inplace_partial_rotary_mul_backward(Tensor(a!) grad, Tensor r1,
  Tensor r2, *, str rotary_mode='interleave', int[2] partial_slice=[0, 0]) -> ()``.
  Both have a CUDA kernel (the library) and a Meta kernel (shape checks
  only, for fake tensors and tracing).  There is no CPU kernel: CPU tensors
  fail in the dispatcher.
* ``partial_slice=None`` means [0, 0], an empty slice (a no-op).
* ``rotary_mode``: "interleave" (the page's only mode: pairs (2i, 2i+1)) or
  "half" (half-split rotate_half: pairs (i, i + L/2)); anything else raises.
* When ``x.requires_grad`` and grad mode is on, the call goes through
  ``InplacePartialRotaryMulFn``: the forward marks x dirty and saves r1 and
  r2; the backward applies the transposed rotation to the incoming
  gradient and returns no gradient for r1 and r2.  As with any in-place op,
  x must not be a leaf that requires grad (use ``y = x * 1.0`` first).
* The backward writes into its own contiguous copy of the incoming gradient,
  so a gradient that autograd also hands to someone else (``retain_grad``,
  an expanded gradient of a sum) is never changed.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import binding

NAMESPACE = "place_partial_rope"
_FWD = "inplace_partial_rotary_mul"
_BWD = "inplace_partial_rotary_mul_backward"
_MODES = ("interleave", "half")

_lib = None


def _check(x: torch.Tensor, rotary_mode: str, partial_slice: Sequence[int]) -> None:
    """The compile-time checks of the page's Meta implementation."""
    if x.dim() != 4:
        raise ValueError(f"inplace_partial_rotary_mul: x must be 4-D (B, S, N, D), got {x.dim()}-D")
    if rotary_mode not in _MODES:
        raise ValueError(f"inplace_partial_rotary_mul: rotary_mode must be 'interleave' or "
                         f"'half', got {rotary_mode!r}")
    if len(partial_slice) != 2:
        raise ValueError(f"inplace_partial_rotary_mul: partial_slice must hold 2 integers, "
                         f"got {len(partial_slice)}")


def _cuda_fwd(x, r1, r2, rotary_mode="interleave", partial_slice=(0, 0)):
    _check(x, rotary_mode, partial_slice)
    binding.rope_partial_inplace_fwd_mode(x, r1, r2, int(partial_slice[0]), int(partial_slice[1]),
                                          rotary_mode)


def _cuda_bwd(grad, r1, r2, rotary_mode="interleave", partial_slice=(0, 0)):
    _check(grad, rotary_mode, partial_slice)
    binding.rope_partial_inplace_bwd_mode(grad, r1, r2, int(partial_slice[0]),
                                          int(partial_slice[1]), rotary_mode)


def _meta(x, r1, r2, rotary_mode="interleave", partial_slice=(0, 0)):
    _check(x, rotary_mode, partial_slice)
    return None


def register() -> None:
    """Define the two operators once per process (idempotent)."""
    global _lib
    if _lib is not None:
        return
    lib = torch.library.Library(NAMESPACE, "DEF")
    lib.define(f"{_FWD}(Tensor(a!) x, Tensor r1, Tensor r2, *, str rotary_mode='interleave', "
               "int[2] partial_slice=[0, 0]) -> ()")
    lib.define(f"{_BWD}(Tensor(a!) grad, Tensor r1, Tensor r2, *, str rotary_mode='interleave', "
               "int[2] partial_slice=[0, 0]) -> ()")
    lib.impl(_FWD, _cuda_fwd, "CUDA")
    lib.impl(_BWD, _cuda_bwd, "CUDA")
    lib.impl(_FWD, _meta, "Meta")
    lib.impl(_BWD, _meta, "Meta")
    _lib = lib


class InplacePartialRotaryMulFn(torch.autograd.Function):
    """Autograd for the in-place rotation: r1 and r2 get no gradient."""

    @staticmethod
    def forward(ctx, x, r1, r2, rotary_mode, partial_slice):
        getattr(torch.ops, NAMESPACE).inplace_partial_rotary_mul(
            x, r1, r2, rotary_mode=rotary_mode, partial_slice=list(partial_slice))
        ctx.mark_dirty(x)
        ctx.save_for_backward(r1, r2)
        ctx.rotary_mode = rotary_mode
        ctx.partial_slice = list(partial_slice)
        return x

    @staticmethod
    def backward(ctx, grad):
        r1, r2 = ctx.saved_tensors
        g = grad.clone(memory_format=torch.contiguous_format)
        getattr(torch.ops, NAMESPACE).inplace_partial_rotary_mul_backward(
            g, r1, r2, rotary_mode=ctx.rotary_mode, partial_slice=ctx.partial_slice)
        return g, None, None, None, None


def inplace_partial_rotary_mul(x: torch.Tensor, r1: torch.Tensor, r2: torch.Tensor, *,
                               rotary_mode: str = "interleave",
                               partial_slice: Optional[Sequence[int]] = None) -> None:
    """Rotate ``x[..., start:end]`` in place (``partial_slice = [start, end]``,
    default empty).  Returns None; x holds the result."""
    register()
    ps = [0, 0] if partial_slice is None else [int(v) for v in partial_slice]
    _check(x, rotary_mode, ps)
    if x.requires_grad and torch.is_grad_enabled():
        InplacePartialRotaryMulFn.apply(x, r1, r2, rotary_mode, ps)
    else:
        getattr(torch.ops, NAMESPACE).inplace_partial_rotary_mul(
            x, r1, r2, rotary_mode=rotary_mode, partial_slice=ps)
    return None

"""GB300-native in-place partial interleaved rotary position embedding.

The compute runs in ``librope_partial.so`` (hand-written sm_103a CUDA
kernels behind a C ABI declared in ``include/rope_partial.h``).  The Python
names below are thin argument marshalling over that library; they raise if
the library has not been built -- there is no CPU fallback.

Submodules:
  binding  -- ctypes binding with the C ABI's names (loaded on first use)
  torch_op -- the PyTorch operator, its Meta kernel and autograd
              (inplace_partial_rotary_mul)
  synth    -- seeded synthetic inputs (no rotation arithmetic)
"""
from __future__ import annotations

_BINDING_NAMES = (
    "rope_partial_inplace_fwd", "rope_partial_inplace_bwd", "rope_partial_inplace_fwd_host",
    "rope_partial_inplace_bwd_host", "prepare_fwd", "prepare_bwd", "RopeError", "load_library",
    "library_path",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    if name in ("inplace_partial_rotary_mul", "InplacePartialRotaryMulFn"):
        from . import torch_op
        return getattr(torch_op, name)
    raise AttributeError(name)

"""ctypes binding of ``librope_partial.so`` (C ABI: ``include/rope_partial.h``).

Argument marshalling only: every step of the operation runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  If the
library has not been built, loading raises -- there is no CPU fallback.

    rope_partial_inplace_fwd(x, r1, r2, start, end, stream=None)
    rope_partial_inplace_bwd(grad, r1, r2, start, end, stream=None)
    rope_partial_inplace_fwd_host(...), rope_partial_inplace_bwd_host(...)   (host tensors)

``x`` / ``grad``: contiguous CUDA tensor (B, S, N, D) of bf16, fp16 or fp32,
modified in place.  ``r1`` (cos) and ``r2`` (sin): 4-D CUDA tensors of the
same dtype and device that broadcast against ``x[..., start:end]`` (any
strides with a contiguous last dim; size-1 dims broadcast).  Both calls are
asynchronous on ``stream`` (default: torch's current stream of x's device).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "librope_partial.so")

ROPE_OK, ROPE_ERR_NULLPTR, ROPE_ERR_INVALID, ROPE_ERR_CUDA = 0, 1, 2, 3
ROPE_BF16, ROPE_FP16, ROPE_FP32 = 0, 1, 2
ROPE_MODE_INTERLEAVE, ROPE_MODE_HALF = 1, 2
MODE_CODE = {"interleave": ROPE_MODE_INTERLEAVE, "half": ROPE_MODE_HALF}
DTYPE_CODE = {torch.bfloat16: ROPE_BF16, torch.float16: ROPE_FP16, torch.float32: ROPE_FP32}

_lib = None


class RopePlan(ctypes.Structure):
    """Mirror of ``rope_plan_t``."""
    _fields_ = [("path", ctypes.c_int32), ("vec_bytes", ctypes.c_int32),
                ("heads_per_thread", ctypes.c_int32), ("threads_per_block", ctypes.c_int32),
                ("blocks", ctypes.c_int64), ("tasks", ctypes.c_int64),
                ("chunks_per_row", ctypes.c_int32), ("r_per_head", ctypes.c_int32),
                ("launches", ctypes.c_int64)]


class RopeTokenRun(ctypes.Structure):
    """Mirror of ``rope_token_run_t``."""
    _fields_ = [("b0", ctypes.c_int64), ("s0", ctypes.c_int64), ("nb", ctypes.c_int64),
                ("ns", ctypes.c_int64)]


class RopeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the CUDA library once; raise if it is missing (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is not built; build it with `python -m place_partial_rope_gb300.build` "
            "(needs nvcc). There is no CPU fallback.")
    lib = ctypes.CDLL(_LIB_PATH)
    i64p = ctypes.POINTER(ctypes.c_int64)
    args = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, i64p, i64p, i64p, i64p,
            ctypes.c_int64, ctypes.c_int64]
    for name in ("rope_partial_inplace_fwd", "rope_partial_inplace_bwd",
                 "rope_partial_inplace_fwd_host", "rope_partial_inplace_bwd_host"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = args + [ctypes.c_void_p]
    for name in ("rope_partial_inplace_fwd_mode", "rope_partial_inplace_bwd_mode"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = args + [ctypes.c_int, ctypes.c_void_p]
    lib.rope_partial_plan_mode.restype = ctypes.c_int
    lib.rope_partial_plan_mode.argtypes = args + [ctypes.c_int, ctypes.c_int32,
                                                  ctypes.POINTER(RopePlan)]
    pos_args = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int] + [ctypes.c_int64] * 4 + \
        [i64p, i64p, ctypes.c_double, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    for name in ("rope_partial_inplace_fwd_pos", "rope_partial_inplace_bwd_pos"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = pos_args
    qk = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_int64] * 10 + [i64p] * 4 + [ctypes.c_void_p]
    for name in ("rope_partial_inplace_fwd_qk", "rope_partial_inplace_bwd_qk"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = qk
    lib.rope_partial_plan.restype = ctypes.c_int
    lib.rope_partial_plan.argtypes = args + [ctypes.c_int32, ctypes.POINTER(RopePlan)]
    lib.rope_partial_token_shard.restype = ctypes.c_int
    lib.rope_partial_token_shard.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                             ctypes.c_int32, i64p, i64p,
                                             ctypes.POINTER(RopeTokenRun), ctypes.POINTER(ctypes.c_int32)]
    lib.rope_status_str.restype = ctypes.c_char_p
    lib.rope_status_str.argtypes = [ctypes.c_int]
    lib.rope_last_error_message.restype = ctypes.c_char_p
    lib.rope_last_error_message.argtypes = []
    _lib = lib
    return lib


def _i64x4(vals):
    return (ctypes.c_int64 * 4)(*[int(v) for v in vals])


def _raise_for(lib, status: int):
    if status != ROPE_OK:
        name = lib.rope_status_str(status).decode()
        msg = lib.rope_last_error_message().decode()
        raise RopeError(status, f"{name}: {msg}")


def _stream_handle(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _marshal(x: torch.Tensor, r1: torch.Tensor, r2: torch.Tensor, host: bool = False):
    if x.dim() != 4:
        raise RopeError(ROPE_ERR_INVALID, f"x must be 4-D (B, S, N, D), got {x.dim()}-D")
    if r1.dim() != 4 or r2.dim() != 4:
        raise RopeError(ROPE_ERR_INVALID, "r1 and r2 must be 4-D")
    if x.dtype not in DTYPE_CODE:
        raise RopeError(ROPE_ERR_INVALID, f"unsupported dtype {x.dtype}")
    if r1.dtype != x.dtype or r2.dtype != x.dtype:
        raise RopeError(ROPE_ERR_INVALID, "r1, r2 and x must share one dtype")
    if not x.is_contiguous():
        raise RopeError(ROPE_ERR_INVALID, "x must be contiguous")
    for t in (x, r1, r2):
        if host and t.is_cuda:
            raise RopeError(ROPE_ERR_INVALID, "the *_host calls take CPU (host) tensors")
        if not host and (not t.is_cuda or t.device != x.device):
            raise RopeError(ROPE_ERR_INVALID, "x, r1 and r2 must be CUDA tensors on one device")
    return (x.data_ptr(), r1.data_ptr(), r2.data_ptr(), DTYPE_CODE[x.dtype], *x.shape,
            _i64x4(r1.shape), _i64x4(r1.stride()), _i64x4(r2.shape), _i64x4(r2.stride()))


def _mode_code(mode) -> int:
    if mode in MODE_CODE:
        return MODE_CODE[mode]
    raise RopeError(ROPE_ERR_INVALID, f"rotary mode {mode!r} is not 'interleave' or 'half'")


def _call(name: str, x, r1, r2, start: int, end: int, stream=None, mode=None) -> None:
    lib = load_library()
    margs = _marshal(x, r1, r2)
    extra = () if mode is None else (_mode_code(mode),)
    with torch.cuda.device(x.device):
        st = getattr(lib, name)(*margs, int(start), int(end), *extra,
                                _stream_handle(stream, x.device))
    _raise_for(lib, st)


def rope_partial_inplace_fwd(x: torch.Tensor, r1: torch.Tensor, r2: torch.Tensor, start: int,
                             end: int, stream=None) -> None:
    """Rotate ``x[..., start:end]`` in place (forward)."""
    _call("rope_partial_inplace_fwd", x, r1, r2, start, end, stream)


def rope_partial_inplace_bwd(grad: torch.Tensor, r1: torch.Tensor, r2: torch.Tensor, start: int,
                             end: int, stream=None) -> None:
    """Overwrite ``grad[..., start:end]`` with the transposed rotation (backward)."""
    _call("rope_partial_inplace_bwd", grad, r1, r2, start, end, stream)


def rope_partial_inplace_fwd_mode(x, r1, r2, start: int, end: int, mode: str = "interleave",
                                  stream=None) -> None:
    """The forward in rotary mode ``"interleave"`` or ``"half"`` (pairs
    (i, i + L/2))."""
    _call("rope_partial_inplace_fwd_mode", x, r1, r2, start, end, stream, mode)


def rope_partial_inplace_bwd_mode(grad, r1, r2, start: int, end: int, mode: str = "interleave",
                                  stream=None) -> None:
    """The backward in rotary mode ``"interleave"`` or ``"half"``."""
    _call("rope_partial_inplace_bwd_mode", grad, r1, r2, start, end, stream, mode)


def _call_host(name: str, x, r1, r2, start: int, end: int, stream=None) -> None:
    lib = load_library()
    margs = _marshal(x, r1, r2, host=True)
    handle = stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else (
        torch.cuda.current_stream().cuda_stream if stream is None else int(stream))
    st = getattr(lib, name)(*margs, int(start), int(end), handle)
    _raise_for(lib, st)


def rope_partial_inplace_fwd_host(x: torch.Tensor, r1: torch.Tensor, r2: torch.Tensor,
                                  start: int, end: int, stream=None) -> None:
    """Forward on host tensors, read and written in place by the GPU (zero
    copy).  x, r1 and r2 are CPU tensors the current CUDA device can reach
    (pinned memory, or any memory on devices with pageable-memory access).
    Asynchronous: synchronise the stream before reading x on the host."""
    _call_host("rope_partial_inplace_fwd_host", x, r1, r2, start, end, stream)


def rope_partial_inplace_bwd_host(grad: torch.Tensor, r1: torch.Tensor, r2: torch.Tensor,
                                  start: int, end: int, stream=None) -> None:
    """Backward on host tensors (zero copy); see rope_partial_inplace_fwd_host."""
    _call_host("rope_partial_inplace_bwd_host", grad, r1, r2, start, end, stream)


def _qk_args(q, k, r1, r2, q_slice, k_slice, stream):
    if q.dim() != 4 or k.dim() != 4:
        raise RopeError(ROPE_ERR_INVALID, "q and k must be 4-D (B, S, N, D)")
    if q.shape[:2] != k.shape[:2]:
        raise RopeError(ROPE_ERR_INVALID, "q and k must share B and S")
    if k.dtype != q.dtype or not k.is_contiguous() or not k.is_cuda or k.device != q.device:
        raise RopeError(ROPE_ERR_INVALID, "k must be a contiguous CUDA tensor of q's dtype and device")
    m = _marshal(q, r1, r2)
    B, S, Nq, Dq = q.shape
    Nk, Dk = k.shape[2], k.shape[3]
    return (q.data_ptr(), k.data_ptr(), r1.data_ptr(), r2.data_ptr(), m[3], B, S, Nq, Dq,
            int(q_slice[0]), int(q_slice[1]), Nk, Dk, int(k_slice[0]), int(k_slice[1]),
            m[8], m[9], m[10], m[11], _stream_handle(stream, q.device))


def rope_partial_inplace_fwd_qk(q, k, r1, r2, q_slice, k_slice, stream=None) -> None:
    """Rotate ``q[..., q_slice]`` and ``k[..., k_slice]`` in place in one
    launch with the same cos/sin rows (shape (B|1, S|1, 1, L))."""
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.rope_partial_inplace_fwd_qk(*_qk_args(q, k, r1, r2, q_slice, k_slice, stream))
    _raise_for(lib, st)


def rope_partial_inplace_bwd_qk(dq, dk, r1, r2, q_slice, k_slice, stream=None) -> None:
    """Backward of rope_partial_inplace_fwd_qk on the two gradients, in place."""
    lib = load_library()
    with torch.cuda.device(dq.device):
        st = lib.rope_partial_inplace_bwd_qk(*_qk_args(dq, dk, r1, r2, q_slice, k_slice, stream))
    _raise_for(lib, st)


def _pos_args(x, positions, start, end, base, mode, stream):
    if x.dim() != 4:
        raise RopeError(ROPE_ERR_INVALID, f"x must be 4-D (B, S, N, D), got {x.dim()}-D")
    if x.dtype not in DTYPE_CODE:
        raise RopeError(ROPE_ERR_INVALID, f"unsupported dtype {x.dtype}")
    if not x.is_contiguous() or not x.is_cuda:
        raise RopeError(ROPE_ERR_INVALID, "x must be a contiguous CUDA tensor")
    if positions.dim() != 2 or positions.dtype != torch.int32:
        raise RopeError(ROPE_ERR_INVALID, "positions must be a 2-D int32 tensor (B|1, S|1)")
    if not positions.is_cuda or positions.device != x.device:
        raise RopeError(ROPE_ERR_INVALID, "positions must be on x's device")
    p_shape = (ctypes.c_int64 * 2)(*positions.shape)
    p_stride = (ctypes.c_int64 * 2)(*positions.stride())
    return (x.data_ptr(), positions.data_ptr(), DTYPE_CODE[x.dtype], *x.shape, p_shape, p_stride,
            float(base), int(start), int(end), _mode_code(mode), _stream_handle(stream, x.device))


def rope_partial_inplace_fwd_pos(x, positions, start: int, end: int, base: float = 10000.0,
                                 mode: str = "interleave", stream=None) -> None:
    """Forward with cos/sin computed in the kernel from int32 positions of
    shape (B|1, S|1): theta_k = p / base^(2k/L)."""
    lib = load_library()
    with torch.cuda.device(x.device):
        st = lib.rope_partial_inplace_fwd_pos(*_pos_args(x, positions, start, end, base, mode, stream))
    _raise_for(lib, st)


def rope_partial_inplace_bwd_pos(grad, positions, start: int, end: int, base: float = 10000.0,
                                 mode: str = "interleave", stream=None) -> None:
    """Backward of rope_partial_inplace_fwd_pos, in place on the gradient."""
    lib = load_library()
    with torch.cuda.device(grad.device):
        st = lib.rope_partial_inplace_bwd_pos(*_pos_args(grad, positions, start, end, base, mode,
                                                          stream))
    _raise_for(lib, st)


def _on_device(dev: int, fn, args) -> int:
    """Call fn(*args) with `dev` as the current CUDA device (the device the
    prepared tensors and stream belong to)."""
    if torch.cuda.current_device() == dev:
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


class PreparedPos:
    """rope_partial_inplace_{fwd,bwd}_pos with arguments marshalled once."""

    def __init__(self, direction: str, x, positions, start, end, base=10000.0, mode="interleave",
                 stream=None):
        self._lib = load_library()
        self._fn = getattr(self._lib, f"rope_partial_inplace_{direction}_pos")
        self._keep = (x, positions)
        self._args = _pos_args(x, positions, start, end, base, mode, stream)
        self._dev = x.device.index

    def __call__(self) -> None:
        st = _on_device(self._dev, self._fn, self._args)
        if st != ROPE_OK:
            _raise_for(self._lib, st)


class PreparedQK:
    """rope_partial_inplace_{fwd,bwd}_qk with arguments marshalled once."""

    def __init__(self, direction: str, q, k, r1, r2, q_slice, k_slice, stream=None):
        self._lib = load_library()
        self._fn = getattr(self._lib, f"rope_partial_inplace_{direction}_qk")
        self._keep = (q, k, r1, r2)
        self._args = _qk_args(q, k, r1, r2, q_slice, k_slice, stream)
        self._dev = q.device.index

    def __call__(self) -> None:
        st = _on_device(self._dev, self._fn, self._args)
        if st != ROPE_OK:
            _raise_for(self._lib, st)


class PreparedCall:
    """One forward or backward call with its arguments marshalled once.

    Calling the object launches the kernel again on the same tensors and
    stream (for loops that launch the same call many times, where per-call
    marshalling would cost more host time than the kernel takes).  It keeps
    references to the tensors so their memory stays alive.
    """

    def __init__(self, name: str, x, r1, r2, start: int, end: int, stream=None, mode=None):
        self._lib = load_library()
        self._fn = getattr(self._lib, name)
        self._keep = (x, r1, r2)
        host = name.endswith("_host")
        dev = torch.device("cuda", torch.cuda.current_device()) if host else x.device
        extra = () if mode is None else (_mode_code(mode),)
        self._args = (*_marshal(x, r1, r2, host=host), int(start), int(end), *extra,
                      _stream_handle(stream, dev))
        self._dev = dev.index if dev.index is not None else torch.cuda.current_device()

    def __call__(self) -> None:
        st = _on_device(self._dev, self._fn, self._args)
        if st != ROPE_OK:
            _raise_for(self._lib, st)


def prepare_fwd(x, r1, r2, start: int, end: int, stream=None, mode=None) -> PreparedCall:
    """``rope_partial_inplace_fwd`` (``_fwd_mode`` when a mode is given) with
    its arguments marshalled once."""
    name = "rope_partial_inplace_fwd" if mode is None else "rope_partial_inplace_fwd_mode"
    return PreparedCall(name, x, r1, r2, start, end, stream, mode)


def prepare_bwd(grad, r1, r2, start: int, end: int, stream=None, mode=None) -> PreparedCall:
    """``rope_partial_inplace_bwd`` (``_bwd_mode`` when a mode is given) with
    its arguments marshalled once."""
    name = "rope_partial_inplace_bwd" if mode is None else "rope_partial_inplace_bwd_mode"
    return PreparedCall(name, grad, r1, r2, start, end, stream, mode)


def prepare_fwd_host(x, r1, r2, start: int, end: int, stream=None) -> PreparedCall:
    """``rope_partial_inplace_fwd_host`` with its arguments marshalled once."""
    return PreparedCall("rope_partial_inplace_fwd_host", x, r1, r2, start, end, stream)


def prepare_bwd_host(grad, r1, r2, start: int, end: int, stream=None) -> PreparedCall:
    """``rope_partial_inplace_bwd_host`` with its arguments marshalled once."""
    return PreparedCall("rope_partial_inplace_bwd_host", grad, r1, r2, start, end, stream)


def rope_partial_plan(x: torch.Tensor, r1: torch.Tensor, r2: torch.Tensor, start: int, end: int,
                      sm_count: int = 0, mode: str = "interleave") -> RopePlan:
    """The launch plan the forward would use (no launch).  Works on CPU
    tensors as well when ``sm_count`` > 0, since only shapes, strides and
    pointer alignment are read."""
    lib = load_library()
    plan = RopePlan()
    args = (x.data_ptr(), r1.data_ptr(), r2.data_ptr(), DTYPE_CODE[x.dtype], *x.shape,
            _i64x4(r1.shape), _i64x4(r1.stride()), _i64x4(r2.shape), _i64x4(r2.stride()))
    st = lib.rope_partial_plan_mode(*args, int(start), int(end), _mode_code(mode), int(sm_count),
                                    ctypes.byref(plan))
    _raise_for(lib, st)
    return plan


def rope_partial_token_shard(B: int, S: int, rank: int, world: int):
    """Rank ``rank`` of ``world``'s tokens of a (B, S) grid: ``(t0, t1, runs)``
    with runs as ``(b0, s0, nb, ns)`` tuples (host only, no CUDA call)."""
    lib = load_library()
    t0, t1, n = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    runs = (RopeTokenRun * 3)()
    st = lib.rope_partial_token_shard(B, S, rank, world, ctypes.byref(t0), ctypes.byref(t1), runs,
                                      ctypes.byref(n))
    _raise_for(lib, st)
    return t0.value, t1.value, [(r.b0, r.s0, r.nb, r.ns) for r in runs[:n.value]]

"""Seeded synthetic inputs for the partial interleaved rotary embedding.

This module only MAKES inputs: activations and gradients drawn from N(0, 1),
position indices, and the cos/sin tables.  It holds none of the rotation's
arithmetic, so the CPU oracle and the CUDA path can both take their inputs
from here without sharing any of the method.

Table recipe ("ANE实战 RoPE位置编码在MIL中的纯ANE实现", section 第一步): for a
position p and pair index i in [0, L/2), theta = p / 10000^(2i/L), where L is
the rotated width (end - start).  cos(theta) and sin(theta) are computed in
float64, rounded once to the storage type, and written to both lanes 2i and
2i+1 (the pair-duplicated layout).

Storage arrays are numpy arrays: float32 for fp32, and uint16 bit patterns
for bf16 and fp16 (numpy has no bfloat16).  The float32 -> bf16/fp16
rounding of the inputs uses torch's CPU conversion (round to nearest even).

The named workloads below are the five shapes the operator is specified on:
a tiny fp32 case, a small-model bf16 forward, a GQA fp16 forward+backward,
an MLA-decode-like query forward (rope part [0, 64) of a 192-wide head), and
a large fp32 case with an unaligned interior slice [34, 98).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

DTYPES = ("bf16", "fp16", "fp32")
ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp32": 4}
TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
BASE = 10000.0


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str
    shape: tuple            # (B, S, N, D) of x
    start: int
    end: int
    r_shape: tuple          # (Br, Sr, Nr, L) of r1 and r2
    positions: str          # "arange" | "per_token_uniform" | "batch_offset"
    pos_max: int            # upper bound of the drawn positions / offsets
    seed: int
    directions: tuple       # ("fwd",) or ("fwd", "bwd")
    description: str

    @property
    def L(self) -> int:
        return self.end - self.start

    @property
    def tokens(self) -> int:
        return self.shape[0] * self.shape[1]

    def slice_elems(self) -> int:
        B, S, N, _ = self.shape
        return B * S * N * self.L

    def algorithmic_bytes(self) -> int:
        """Slice bytes read + written, plus the unique cos and sin bytes."""
        e = ELEM_BYTES[self.dtype]
        r_elems = int(np.prod(self.r_shape))
        return 2 * self.slice_elems() * e + 2 * r_elems * e


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", "fp32", (1, 16, 2, 64), 0, 32, (1, 16, 1, 32), "arange", 0, 1000,
                 ("fwd", "bwd"), "tiny fp32 (1,16,2,64) slice [0,32), r (1,16,1,32)"),
        Workload("small_model", "bf16", (16, 256, 12, 64), 0, 64, (1, 256, 1, 64), "arange", 0,
                 1001, ("fwd",), "small-model bf16 (16,256,12,64) full slice, r (1,256,1,64)"),
        Workload("gqa", "fp16", (32, 2048, 16, 128), 0, 64, (1, 2048, 1, 64), "arange", 0, 1002,
                 ("fwd", "bwd"), "GQA fp16 (32,2048,16,128) slice [0,64), r (1,2048,1,64)"),
        Workload("mla_decode_q", "bf16", (4096, 1, 128, 192), 0, 64, (4096, 1, 1, 64),
                 "per_token_uniform", 32768, 1003, ("fwd",),
                 "MLA-decode query bf16 (4096,1,128,192) slice [0,64), r (4096,1,1,64)"),
        Workload("large_unaligned", "fp32", (4, 8192, 32, 128), 34, 98, (4, 8192, 1, 64),
                 "batch_offset", 4096, 1004, ("fwd", "bwd"),
                 "large fp32 (4,8192,32,128) unaligned slice [34,98), r (4,8192,1,64)"),
    ]
}


# The query workload above plus its key: in MLA decoding the rope part of
# the key is one (T, 64) row per token, rotated with the same cos/sin row as
# the query's rope lanes [0, 64) of each 192-wide head.
QK_KEY_SHAPE = (4096, 1, 1, 64)
QK_KEY_SLICE = (0, 64)
QK_KEY_SEED = 1603


def qk_inputs(with_grad: bool = False):
    """q, k, r1, r2 (and dq, dk) of the fused query + key MLA-decode case."""
    w = WORKLOADS["mla_decode_q"]
    q, r1, r2, _ = workload_inputs(w, with_grad=False)
    k = normal(QK_KEY_SHAPE, w.dtype, QK_KEY_SEED)
    if not with_grad:
        return q, k, r1, r2
    dq = normal(w.shape, w.dtype, w.seed + 500)
    dk = normal(QK_KEY_SHAPE, w.dtype, QK_KEY_SEED + 500)
    return q, k, r1, r2, dq, dk


def qk_algorithmic_bytes() -> int:
    """Slice bytes of q and k read + written, plus the unique cos/sin bytes."""
    w = WORKLOADS["mla_decode_q"]
    e = ELEM_BYTES[w.dtype]
    k_elems = int(np.prod(QK_KEY_SHAPE[:3])) * (QK_KEY_SLICE[1] - QK_KEY_SLICE[0])
    return w.algorithmic_bytes() + 2 * k_elems * e


# --------------------------------------------------------------------------
# storage conversions (input side only)
# --------------------------------------------------------------------------

def to_storage(a, dtype: str) -> np.ndarray:
    """float32/float64 values -> storage array (RNE), via numpy / torch CPU."""
    if dtype == "fp32":
        return np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    if dtype == "fp16":
        return np.ascontiguousarray(np.asarray(a).astype(np.float16)).view(np.uint16)
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float64)))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Storage array -> CPU torch tensor of the storage dtype (shares memory)."""
    if dtype == "fp32":
        return torch.from_numpy(a)
    if dtype == "fp16":
        return torch.from_numpy(a.view(np.float16))
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)


def from_torch(t: torch.Tensor) -> np.ndarray:
    """CPU/GPU torch tensor -> storage array on the host (a copy)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------

def normal(shape, dtype: str, seed: int) -> np.ndarray:
    """Seeded N(0,1) values drawn in float32, rounded to the storage type."""
    rng = np.random.default_rng(seed)
    return to_storage(rng.standard_normal(size=shape, dtype=np.float32), dtype)


def positions(w: Workload) -> np.ndarray:
    """Integer positions of shape r_shape[:3] for a named workload."""
    Br, Sr, Nr, _ = w.r_shape
    rng = np.random.default_rng(w.seed + 250)
    if w.positions == "arange":
        p = np.broadcast_to(np.arange(Sr, dtype=np.int64)[None, :, None], (Br, Sr, Nr))
    elif w.positions == "per_token_uniform":
        p = rng.integers(0, w.pos_max, size=(Br, Sr, Nr), dtype=np.int64)
    elif w.positions == "batch_offset":
        off = rng.integers(0, w.pos_max, size=(Br,), dtype=np.int64)
        p = off[:, None, None] + np.arange(Sr, dtype=np.int64)[None, :, None]
        p = np.broadcast_to(p, (Br, Sr, Nr))
    else:
        raise ValueError(w.positions)
    return np.ascontiguousarray(p)


def rope_table(pos: np.ndarray, L: int, dtype: str, base: float = BASE,
               layout: str = "interleave"):
    """cos/sin tables of shape pos.shape + (L,): pair i's value in lanes 2i
    and 2i+1 (``layout="interleave"``), or in lanes i and i + L/2
    (``layout="half"``, the layout of the half-split mode)."""
    i = np.arange(L // 2, dtype=np.float64)
    inv = base ** (-(2.0 * i) / L)
    theta = pos.astype(np.float64)[..., None] * inv
    if layout == "half":
        c = np.concatenate([np.cos(theta)] * 2, axis=-1)
        s = np.concatenate([np.sin(theta)] * 2, axis=-1)
    else:
        c = np.repeat(np.cos(theta), 2, axis=-1)
        s = np.repeat(np.sin(theta), 2, axis=-1)
    return to_storage(c, dtype), to_storage(s, dtype)


def random_table(shape, dtype: str, seed: int):
    """Independent N(0,1) cos and sin stand-ins (the pages' randn examples):
    neither pair-duplicated nor orthogonal, so they exercise every lane."""
    rng = np.random.default_rng(seed)
    c = rng.standard_normal(size=shape, dtype=np.float32)
    s = rng.standard_normal(size=shape, dtype=np.float32)
    return to_storage(c, dtype), to_storage(s, dtype)


def workload_inputs(w: Workload, with_grad: bool = True):
    """x, r1, r2 (and grad when the workload has a backward) for a named workload."""
    x = normal(w.shape, w.dtype, w.seed)
    r1, r2 = rope_table(positions(w), w.L, w.dtype)
    g = normal(w.shape, w.dtype, w.seed + 500) if (with_grad and "bwd" in w.directions) else None
    return x, r1, r2, g


BROADCAST_FORMS = {
    # name -> which of (B, S, N) the cos/sin tensors keep (others are size 1)
    "BSND": (1, 1, 1), "B1ND": (1, 0, 1), "B11D": (1, 0, 0), "111D": (0, 0, 0),
    "BS1D": (1, 1, 0), "1S1D": (0, 1, 0), "1SND": (0, 1, 1), "11ND": (0, 0, 1),
}


def r_shape_for(form: str, shape, L: int):
    keep = BROADCAST_FORMS[form]
    return tuple(shape[k] if keep[k] else 1 for k in range(3)) + (L,)


def case(shape, start: int, end: int, dtype: str, form: str = "BS1D", seed: int = 0,
         table: str = "random", layout: str = "interleave"):
    """A small seeded case: x, r1, r2, grad for arbitrary shapes and forms."""
    L = end - start
    rs = r_shape_for(form, shape, L)
    x = normal(shape, dtype, seed)
    g = normal(shape, dtype, seed + 500)
    if table == "random":
        r1, r2 = random_table(rs, dtype, seed + 77)
    else:
        pos = np.broadcast_to(np.arange(rs[1], dtype=np.int64)[None, :, None] +
                              np.arange(rs[0], dtype=np.int64)[:, None, None] * 3 +
                              np.arange(rs[2], dtype=np.int64)[None, None, :] * 5, rs[:3])
        r1, r2 = rope_table(np.ascontiguousarray(pos), L, dtype, layout=layout)
    return x, r1, r2, g

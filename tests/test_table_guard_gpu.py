"""cos/sin reads stay inside the table: r1 and r2 are views into buffers
filled with NaN around them (one extra index on each side of every dim,
extra lanes past each row), so any read outside the view's own elements
turns into a NaN in the output, which the bit-exact comparison with the
oracle (run on the clean tables) catches.  Every kernel kind that reads a
table runs: interleave, half-split with the partner in another lane and in
the same thread, the element paths, and the fused query + key call."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, assert_same, to_dev
from place_partial_rope_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def poisoned_view(r: np.ndarray, dtype: str) -> torch.Tensor:
    """r as a strided view whose every neighbour in the buffer is NaN; the
    view starts on a 16-byte boundary and its row pitch keeps it there."""
    e = synth.ELEM_BYTES[dtype]
    k = 16 // e                       # lanes of padding before each row
    Br, Sr, Nr, L = r.shape
    pitch = -(-(L + 2 * k) // k) * k  # row pitch in elements, a multiple of 16 bytes
    T = synth.TORCH_DTYPE[dtype]
    big = torch.full((Br + 2, Sr + 2, Nr + 2, pitch), float("nan"), dtype=T, device=DEV)
    view = big[1:1 + Br, 1:1 + Sr, 1:1 + Nr, k:k + L]
    view.copy_(to_dev(r, dtype))
    assert view.data_ptr() % 16 == 0 and view.stride()[3] == 1
    return view


CASES = [
    ((2, 5, 3, 64), 0, 64), ((2, 5, 3, 64), 8, 40), ((2, 5, 3, 64), 2, 58), ((2, 5, 3, 64), 3, 61),
    ((3, 4, 7, 48), 1, 3), ((2, 3, 13, 24), 6, 22), ((4, 9, 1, 10), 0, 10), ((2, 3, 5, 128), 34, 98),
    ((1, 3, 4, 96), 0, 96), ((2, 3, 6, 64), 0, 48),
]
FORMS = ["BS1D", "B11D", "1S1D", "111D", "BSND", "1SND", "B1ND"]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("mode", ["interleave", "half"])
@pytest.mark.parametrize("k", range(len(CASES)))
def test_reads_stay_inside_the_tables(dtype, mode, k):
    shape, st, en = CASES[k]
    for f, form in enumerate(FORMS):
        x, r1, r2, g = synth.case(shape, st, en, dtype, form, seed=900 + 10 * k + f, layout=mode)
        c, s = poisoned_view(r1, dtype), poisoned_view(r2, dtype)
        for direction, inp in (("fwd", x), ("bwd", g)):
            xd = to_dev(inp, dtype)
            fn = binding.rope_partial_inplace_fwd_mode if direction == "fwd" else binding.rope_partial_inplace_bwd_mode
            fn(xd, c, s, st, en, mode)
            torch.cuda.synchronize()
            ofn = oracle.fwd if direction == "fwd" else oracle.bwd
            want = ofn(inp, r1, r2, dtype, st, en, oracle.GATHER_CHAIN, mode)
            assert_same(synth.from_torch(xd), want, dtype, f"{shape} [{st},{en}) {form} {mode} {direction}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_fused_query_key_reads_stay_inside_the_table(dtype):
    q, r1, r2, dq = synth.case((3, 5, 8, 96), 0, 64, dtype, "BS1D", seed=950)
    k = synth.normal((3, 5, 2, 80), dtype, 951)
    c, s = poisoned_view(r1, dtype), poisoned_view(r2, dtype)
    qd, kd = to_dev(q, dtype), to_dev(k, dtype)
    binding.rope_partial_inplace_fwd_qk(qd, kd, c, s, (0, 64), (8, 72))
    torch.cuda.synchronize()
    wq, wk = oracle.rope_qk(oracle.FWD, q, k, r1, r2, dtype, (0, 64), (8, 72))
    assert_same(synth.from_torch(qd), wq, dtype, "query")
    assert_same(synth.from_torch(kd), wk, dtype, "key")

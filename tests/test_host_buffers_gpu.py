"""GPU parity of the host-buffer entry points (zero copy): the kernel reads
and writes page-locked host tensors in place.  Same bar as the device path:
bit-exact against the CPU oracle, untouched bytes unchanged."""
import numpy as np
import pytest
import torch

from gpu_util import DEV, assert_same, run_oracle, to_dev
from place_partial_rope_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def run_host(direction, x, r1, r2, dtype, start, end, pin=True, r_on_device=False):
    xt = synth.to_torch(np.ascontiguousarray(x).copy(), dtype)
    ct = synth.to_torch(np.ascontiguousarray(r1), dtype)
    st = synth.to_torch(np.ascontiguousarray(r2), dtype)
    if pin:
        xt, ct, st = xt.pin_memory(), ct.pin_memory(), st.pin_memory()
    if r_on_device:
        ct, st = ct.to(DEV), st.to(DEV)
    fn = binding.rope_partial_inplace_fwd_host if direction == "fwd" else binding.rope_partial_inplace_bwd_host
    if r_on_device:
        # cos/sin in device memory, x on the host: the raw C call takes any mix
        lib = binding.load_library()
        args = (xt.data_ptr(), ct.data_ptr(), st.data_ptr(), binding.DTYPE_CODE[xt.dtype], *xt.shape,
                binding._i64x4(ct.shape), binding._i64x4(ct.stride()), binding._i64x4(st.shape),
                binding._i64x4(st.stride()), start, end, torch.cuda.current_stream().cuda_stream)
        name = "rope_partial_inplace_fwd_host" if direction == "fwd" else "rope_partial_inplace_bwd_host"
        assert getattr(lib, name)(*args) == binding.ROPE_OK, lib.rope_last_error_message()
    else:
        fn(xt, ct, st, start, end)
    torch.cuda.synchronize()
    return synth.from_torch(xt)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("shape,st,en,form", [((2, 5, 3, 64), 0, 64, "BS1D"),
                                              ((2, 5, 3, 64), 34, 62, "BSND"),
                                              ((3, 7, 5, 40), 3, 37, "1S1D"),
                                              ((1, 300, 4, 128), 0, 64, "1S1D"),
                                              ((2, 37, 3, 66), 1, 65, "BS1D"),   # odd start, 32 pairs
                                              ((4, 50, 2, 128), 32, 96, "BS1D")])  # mid-row slice
def test_pinned_host_buffers(dtype, shape, st, en, form):
    x, r1, r2, g = synth.case(shape, st, en, dtype, form, seed=41)
    for direction, inp in (("fwd", x), ("bwd", g)):
        got = run_host(direction, inp, r1, r2, dtype, st, en)
        assert_same(got, run_oracle(direction, inp, r1, r2, dtype, st, en), dtype, f"host {direction}")


def test_host_x_with_device_tables():
    x, r1, r2, g = synth.case((2, 9, 4, 48), 8, 40, "bf16", "BS1D", seed=43)
    got = run_host("fwd", x, r1, r2, "bf16", 8, 40, r_on_device=True)
    assert_same(got, run_oracle("fwd", x, r1, r2, "bf16", 8, 40), "bf16", "host x, device cos/sin")


@pytest.mark.parametrize("name,direction", [("gqa", "bwd"), ("large_unaligned", "fwd"),
                                            ("large_unaligned", "bwd")])
def test_named_workload_on_host_buffers(name, direction):
    """Full size on page-locked host buffers, every element: the gqa shape
    and the large fp32 shape, whose calls the benchmark's end-to-end figure
    times."""
    w = synth.WORKLOADS[name]
    x, r1, r2, g = synth.workload_inputs(w)
    inp = x if direction == "fwd" else g
    got = run_host(direction, inp, r1, r2, w.dtype, w.start, w.end)
    assert_same(got, run_oracle(direction, inp, r1, r2, w.dtype, w.start, w.end), w.dtype,
                f"{name} {direction} host")


def test_pageable_host_memory_is_used_or_refused():
    """Ordinary (pageable) host memory: devices that can reach it (pageable
    memory access, e.g. through the coherent CPU link) compute the right
    answer; other devices get ROPE_ERR_INVALID before any launch."""
    x, r1, r2, _ = synth.case((2, 4, 3, 32), 0, 32, "fp32", "BS1D", seed=47)
    try:
        got = run_host("fwd", x, r1, r2, "fp32", 0, 32, pin=False)
    except binding.RopeError as e:
        assert e.status == binding.ROPE_ERR_INVALID and "pageable" in str(e)
        return
    assert_same(got, run_oracle("fwd", x, r1, r2, "fp32", 0, 32), "fp32", "pageable host")


def test_host_calls_reject_device_tensors():
    x, r1, r2, _ = synth.case((1, 2, 2, 8), 0, 8, "fp32", "BS1D", seed=1)
    with pytest.raises(binding.RopeError):
        binding.rope_partial_inplace_fwd_host(to_dev(x, "fp32"), to_dev(r1, "fp32"), to_dev(r2, "fp32"), 0, 8)

"""The PyTorch operator and autograd on the GPU, against the CPU oracle.

Follows the single-op and training examples of "CANN ops-transformer
inplace_partial_rotary_mul" (sections 单算子模式调用 and 训练模式调用: B=2,
S=32, N=8, D=128, fp16, partial_slice [0, 64), r1/r2 randn of shape
(B, S, 1, 64); y = x * 1.0; the op on y; y.sum().backward()).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, assert_same, to_dev
from place_partial_rope_gb300 import synth, torch_op

pytestmark = pytest.mark.gpu

SHAPE, START, END = (2, 32, 8, 128), 0, 64


def inputs(dtype="fp16", seed=3):
    return synth.case(SHAPE, START, END, dtype, "BS1D", seed=seed)


@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
def test_single_op_matches_oracle(dtype):
    x, r1, r2, _ = inputs(dtype)
    xd = to_dev(x, dtype)
    out = torch_op.inplace_partial_rotary_mul(xd, to_dev(r1, dtype), to_dev(r2, dtype),
                                              rotary_mode="interleave", partial_slice=[START, END])
    assert out is None
    torch.cuda.synchronize()
    assert_same(synth.from_torch(xd), oracle.fwd(x, r1, r2, dtype, START, END), dtype, "op fwd")


def test_default_slice_is_a_noop():
    x, r1, r2, _ = inputs()
    xd = to_dev(x, "fp16")
    empty = torch.empty((1, 1, 1, 0), dtype=torch.float16, device=DEV)
    torch_op.inplace_partial_rotary_mul(xd, empty, empty)  # partial_slice None -> [0, 0]
    torch.cuda.synchronize()
    assert_same(synth.from_torch(xd), x, "fp16", "no-op")


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_training_autograd(dtype):
    """x.grad equals the oracle's backward of the upstream gradient; y.grad
    (retained) is not changed by the in-place backward; r1/r2 get None."""
    x, r1, r2, g = inputs(dtype, seed=5)
    xd = to_dev(x, dtype).requires_grad_(True)
    c = to_dev(r1, dtype).requires_grad_(True)
    s = to_dev(r2, dtype).requires_grad_(True)
    w = to_dev(g, dtype)
    y = xd * 1.0
    y.retain_grad()
    torch_op.inplace_partial_rotary_mul(y, c, s, rotary_mode="interleave", partial_slice=[START, END])
    assert y.grad_fn is not None
    loss = (y * w).sum()
    loss.backward()
    torch.cuda.synchronize()
    assert c.grad is None and s.grad is None
    assert_same(synth.from_torch(y.grad), g, dtype, "y.grad untouched")
    assert_same(synth.from_torch(xd.grad), oracle.bwd(g, r1, r2, dtype, START, END), dtype, "x.grad")
    # the forward value seen through autograd is the oracle's forward
    assert_same(synth.from_torch(y.detach()), oracle.fwd(x, r1, r2, dtype, START, END), dtype, "y")


def test_sum_backward_with_expanded_gradient():
    x, r1, r2, _ = inputs(seed=9)
    xd = to_dev(x, "fp16").requires_grad_(True)
    y = xd * 1.0
    torch_op.inplace_partial_rotary_mul(y, to_dev(r1, "fp16"), to_dev(r2, "fp16"),
                                        partial_slice=[START, END])
    y.sum().backward()  # the incoming gradient is an expanded (stride-0) tensor of ones
    ones = synth.to_storage(np.ones(SHAPE), "fp16")
    assert_same(synth.from_torch(xd.grad), oracle.bwd(ones, r1, r2, "fp16", START, END), "fp16",
                "grad of sum")


def test_leaf_requiring_grad_is_rejected():
    x, r1, r2, _ = inputs()
    xd = to_dev(x, "fp16").requires_grad_(True)
    with pytest.raises(RuntimeError):
        torch_op.inplace_partial_rotary_mul(xd, to_dev(r1, "fp16"), to_dev(r2, "fp16"),
                                            partial_slice=[START, END])


def test_traced_by_torch_compile():
    """Graph capture through the Meta kernel (torch.compile with the
    aot_eager backend, full graph): same result as the eager call."""
    x, r1, r2, _ = inputs(seed=13)
    c, s = to_dev(r1, "fp16"), to_dev(r2, "fp16")

    def f(t):
        y = t * 1.0
        torch.ops.place_partial_rope.inplace_partial_rotary_mul(y, c, s, partial_slice=[START, END])
        return y

    torch_op.register()
    compiled = torch.compile(f, backend="aot_eager", fullgraph=True)
    got = compiled(to_dev(x, "fp16"))
    torch.cuda.synchronize()
    assert_same(synth.from_torch(got), oracle.fwd(x, r1, r2, "fp16", START, END), "fp16", "compiled")

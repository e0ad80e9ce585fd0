"""The PyTorch operator without a GPU: schema, the Meta checks of the page's
graph-mode support ("CANN ops-transformer inplace_partial_rotary_mul",
section 图模式调用: errors for x.dim() != 4, rotary_mode != 'interleave' and
len(partial_slice) != 2), the None -> [0, 0] default, and no CPU kernel."""
import pytest
import torch

from place_partial_rope_gb300 import torch_op


def setup_module():
    torch_op.register()
    torch_op.register()  # idempotent


def test_schema_matches_the_page():
    op = torch.ops.place_partial_rope.inplace_partial_rotary_mul.default
    s = str(op._schema)
    # torch prints an int[2] default of [0, 0] in its broadcast form "0"
    want = ("place_partial_rope::inplace_partial_rotary_mul(Tensor(a!) x, Tensor r1, Tensor r2, *, "
            "str rotary_mode=\"interleave\", int[2] partial_slice={}) -> ()")
    assert s in (want.format("[0, 0]"), want.format("0"))
    assert op._schema.arguments[4].default_value in ([0, 0], 0)
    b = str(torch.ops.place_partial_rope.inplace_partial_rotary_mul_backward.default._schema)
    assert "Tensor(a!) grad" in b


def meta(*shape):
    return torch.empty(shape, device="meta", dtype=torch.float16)


def test_meta_kernel_accepts_valid_calls():
    x, r = meta(2, 4, 3, 16), meta(1, 4, 1, 8)
    torch.ops.place_partial_rope.inplace_partial_rotary_mul(x, r, r, partial_slice=[0, 8])
    torch.ops.place_partial_rope.inplace_partial_rotary_mul_backward(x, r, r, partial_slice=[0, 8])
    torch_op.inplace_partial_rotary_mul(x, r, r)  # None -> [0, 0]


@pytest.mark.parametrize("x,mode,ps,needle", [
    (meta(2, 4, 16), "interleave", [0, 8], "4-D"),
    (meta(1, 2, 4, 3, 16), "interleave", [0, 8], "4-D"),
    (meta(2, 4, 3, 16), "neox", [0, 8], "interleave"),
    (meta(2, 4, 3, 16), "interleave", [0, 8, 2], "2 integers"),
    (meta(2, 4, 3, 16), "interleave", [4], "2 integers"),
])
def test_meta_checks_raise(x, mode, ps, needle):
    r = meta(1, 4, 1, 8)
    with pytest.raises((ValueError, RuntimeError), match=needle):
        torch_op.inplace_partial_rotary_mul(x, r, r, rotary_mode=mode, partial_slice=ps)


def test_no_cpu_kernel():
    x, r = torch.zeros(2, 4, 3, 16), torch.zeros(1, 4, 1, 8)
    with pytest.raises((NotImplementedError, RuntimeError)):
        torch_op.inplace_partial_rotary_mul(x, r, r, partial_slice=[0, 8])

"""GPU parity of the fused query + key call against its definition (the
oracle applied to q and to k with the same cos/sin rows), bit for bit.

The MLA case follows "ascend-transformer-boost MlaPreprocessOperation"
(sections 3 and 4: RoPE on Q[..., :qRopeDim] and K[..., :kRopeDim] with
qRopeDim = kRopeDim = 64, cos/sin of shape [tokenNum, 64])."""
import pytest
import torch

import oracle
from gpu_util import DEV, assert_same, to_dev
from place_partial_rope_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def run(direction, q, k, r1, r2, dtype, qs, ks):
    qd, kd = to_dev(q, dtype), to_dev(k, dtype)
    fn = binding.rope_partial_inplace_fwd_qk if direction == "fwd" else binding.rope_partial_inplace_bwd_qk
    fn(qd, kd, to_dev(r1, dtype), to_dev(r2, dtype), qs, ks)
    torch.cuda.synchronize()
    return synth.from_torch(qd), synth.from_torch(kd)


def check(direction, q, k, r1, r2, dtype, qs, ks, what):
    gq, gk = run(direction, q, k, r1, r2, dtype, qs, ks)
    d = oracle.FWD if direction == "fwd" else oracle.BWD
    wq, wk = oracle.rope_qk(d, q, k, r1, r2, dtype, qs, ks)
    assert_same(gq, wq, dtype, f"{what} q {direction}")
    assert_same(gk, wk, dtype, f"{what} k {direction}")


@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_mla_decode_query_and_key_full_size(direction):
    q, k, r1, r2, dq, dk = synth.qk_inputs(with_grad=True)
    a, b = (q, k) if direction == "fwd" else (dq, dk)
    check(direction, a, b, r1, r2, "bf16", synth.QK_KEY_SLICE, synth.QK_KEY_SLICE, "mla")


@pytest.mark.parametrize("direction", ["fwd", "bwd"])
def test_gqa_query_and_key_full_size(direction):
    """The GQA pair the benchmark times: the gqa query (32,2048,16,128) and
    4 key heads of the same rows, slices [0, 64), fp16, one cos/sin row per
    position shared by every batch; every element."""
    g = synth.WORKLOADS["gqa"]
    seed = g.seed + (0 if direction == "fwd" else 500)
    q = synth.normal(g.shape, g.dtype, seed)
    k = synth.normal(g.shape[:2] + (4,) + g.shape[3:], g.dtype, g.seed + 600)
    r1, r2 = synth.rope_table(synth.positions(g), g.L, g.dtype)
    check(direction, q, k, r1, r2, g.dtype, (g.start, g.end), (g.start, g.end), "gqa")


CASES = [
    # (B, S), (Nq, Dq, qs, qe), (Nk, Dk, ks, ke), broadcast of cos/sin over (B, S)
    ((2, 5), (3, 64, 0, 32), (2, 48, 16, 48), (1, 1)),
    ((3, 4), (8, 192, 0, 64), (1, 64, 0, 64), (1, 0)),
    ((2, 6), (5, 40, 3, 23), (4, 24, 1, 21), (1, 1)),      # odd starts: scalar pairs
    ((1, 9), (16, 128, 2, 66), (2, 64, 0, 64), (0, 1)),    # 4-byte offset for the query
    ((4, 3), (7, 64, 0, 64), (0, 64, 0, 64), (1, 1)),      # no key heads: query only
]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("k_", range(len(CASES)))
def test_fused_cases(dtype, k_):
    (B, S), (Nq, Dq, qs, qe), (Nk, Dk, ks, ke), (kb, ks_) = CASES[k_]
    L = qe - qs
    q = synth.normal((B, S, Nq, Dq), dtype, 500 + k_)
    k = synth.normal((B, S, Nk, Dk), dtype, 600 + k_)
    r1, r2 = synth.random_table((B if kb else 1, S if ks_ else 1, 1, L), dtype, 700 + k_)
    for direction in ("fwd", "bwd"):
        check(direction, q, k, r1, r2, dtype, (qs, qe), (ks, ke), f"case {k_}")


def test_fused_equals_two_single_launches():
    q, k, r1, r2 = synth.qk_inputs()
    qd, kd = to_dev(q, "bf16"), to_dev(k, "bf16")
    c, s = to_dev(r1, "bf16"), to_dev(r2, "bf16")
    q2, k2 = qd.clone(), kd.clone()
    binding.rope_partial_inplace_fwd_qk(qd, kd, c, s, (0, 64), (0, 64))
    binding.rope_partial_inplace_fwd(q2, c, s, 0, 64)
    binding.rope_partial_inplace_fwd(k2, c, s, 0, 64)
    torch.cuda.synchronize()
    assert torch.equal(qd.view(torch.int16), q2.view(torch.int16))
    assert torch.equal(kd.view(torch.int16), k2.view(torch.int16))


def test_fused_call_split_into_several_launches():
    """Query and key of one pair per row over 2^30 + 3 tokens each: 2^31 + 6
    work items, so the fused call runs as two launches, each covering the
    query's items of its tokens, then the key's.  With cos = 0 and sin = 1
    the forward is the exact quarter turn (a, b) -> (-b, a) at any size; rows
    at the start, at the launch boundary and at the end are also checked
    against the oracle with a random table."""
    S = 2**30 + 3
    g = torch.Generator(device=DEV).manual_seed(4321)
    q = torch.randn((1, S, 1, 2), generator=g, device=DEV, dtype=torch.float32).to(torch.float16)
    k = torch.randn((1, S, 1, 4), generator=g, device=DEV, dtype=torch.float32).to(torch.float16)
    zero = torch.zeros((1, 1, 1, 2), dtype=torch.float16, device=DEV)
    one = torch.ones((1, 1, 1, 2), dtype=torch.float16, device=DEV)
    q0, k0 = q.clone(), k.clone()
    binding.rope_partial_inplace_fwd_qk(q, k, zero, one, (0, 2), (2, 4))
    torch.cuda.synchronize()
    assert torch.equal(q[..., 0], -q0[..., 1]) and torch.equal(q[..., 1], q0[..., 0])
    assert torch.equal(k[..., 2], -k0[..., 3]) and torch.equal(k[..., 3], k0[..., 2])
    assert torch.equal(k[..., :2], k0[..., :2])
    c_h, s_h = synth.random_table((1, 1, 1, 2), "fp16", 19)
    q2, k2 = q0.clone(), k0.clone()
    binding.rope_partial_inplace_fwd_qk(q2, k2, to_dev(c_h, "fp16"), to_dev(s_h, "fp16"), (0, 2), (2, 4))
    torch.cuda.synchronize()
    for t0 in (0, 2**30 - 2, S - 3):
        qi = synth.from_torch(q0[:, t0:t0 + 3])
        ki = synth.from_torch(k0[:, t0:t0 + 3])
        wq, wk = oracle.rope_qk(oracle.FWD, qi, ki, c_h, s_h, "fp16", (0, 2), (2, 4))
        assert_same(synth.from_torch(q2[:, t0:t0 + 3]), wq, "fp16", f"query rows at {t0}")
        assert_same(synth.from_torch(k2[:, t0:t0 + 3]), wk, "fp16", f"key rows at {t0}")
    del q, k, q0, k0, q2, k2
    torch.cuda.empty_cache()

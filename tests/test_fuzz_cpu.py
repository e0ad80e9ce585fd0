"""The fuzz draws on the CPU: every draw is a valid call, and the table draws
reach every kernel path and access width, so the GPU fuzz test exercises
them all.  Plans are queried with an explicit SM count on host tensors laid
out as the GPU test lays them out (only shapes, strides and pointer
alignment are read)."""
import collections

import pytest
import torch

import fuzz_cases as fc
from place_partial_rope_gb300 import binding, build, synth
from test_fuzz_gpu import GUARD, N_POS, N_QK, N_TABLE

SM_COUNT = 152


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.load_library()


def host_plan(c: fc.TableCase):
    td = synth.TORCH_DTYPE[c.dtype]
    n = int(torch.Size(c.shape).numel())
    x = torch.empty(c.x_offset + n + GUARD, dtype=td)[c.x_offset:c.x_offset + n].view(c.shape)
    rs = synth.r_shape_for(c.form, c.shape, c.sl.L)
    padded = torch.empty(rs[:3] + (c.sl.L + c.r_pad,), dtype=td)
    r = padded[..., c.r_offset:c.r_offset + c.sl.L]
    return binding.rope_partial_plan(x, r, r, c.sl.start, c.sl.end, SM_COUNT, c.mode)


def test_table_draws_reach_every_path():
    paths = collections.Counter()
    widths = collections.Counter()
    for k in range(N_TABLE):
        c = fc.table_case(k)
        plan = host_plan(c)
        paths[plan.path] += 1
        if plan.path:
            widths[plan.vec_bytes] += 1
    # 0 = nothing to do, 1 = vector accesses, 2 = element pairs,
    # 3 = half-split lanes, 4 = odd start with a lane per aligned vector
    assert set(paths) == {0, 1, 2, 3, 4}, paths
    assert {4, 8, 16} <= set(widths), widths
    assert min(paths[p] for p in (1, 2, 3, 4)) >= 8, paths


def test_odd_start_draws_reach_every_vector_width():
    """The odd-start kernel is drawn for every storage type and vector
    width, on rows that straddle warps and rows that do not."""
    seen, straddle = collections.Counter(), 0
    for k in range(N_TABLE):
        c = fc.table_case(k)
        plan = host_plan(c)
        if plan.path != 4:
            continue
        seen[(synth.ELEM_BYTES[c.dtype], plan.vec_bytes)] += 1
        straddle += 32 % plan.chunks_per_row != 0
    assert set(seen) == {(2, 16), (2, 8), (4, 16), (4, 8)}, seen
    assert straddle >= 8, straddle


def test_draws_are_valid_and_varied():
    modes, dtypes, odd = collections.Counter(), collections.Counter(), 0
    for k in range(N_TABLE):
        c = fc.table_case(k)
        D, st, en = c.sl.D, c.sl.start, c.sl.end
        assert c.shape[3] == D and 0 <= st <= en <= D and (en - st) % 2 == 0 and D % 2 == 0
        assert 0 <= c.r_offset <= c.r_pad and int(torch.Size(c.shape).numel()) <= fc.MAX_ELEMS
        modes[c.mode] += 1
        dtypes[c.dtype] += 1
        odd += st % 2
    assert set(modes) == {"interleave", "half"} and set(dtypes) == set(synth.DTYPES)
    assert odd >= N_TABLE // 5
    for k in range(N_QK):
        c = fc.qk_case(k)
        (_, Dq, qs, qe), (_, Dk, ks, ke) = c.q, c.k
        assert qe - qs == ke - ks and 0 <= qs <= qe <= Dq and 0 <= ks <= ke <= Dk
        assert synth.BROADCAST_FORMS[c.form][2] == 0
    for k in range(N_POS):
        c = fc.pos_case(k)
        assert c.pos_shape[0] in (1, c.shape[0]) and c.pos_shape[1] in (1, c.shape[1])


def test_plans_of_the_draws_keep_their_contract():
    """For every table draw: the work items cover each row's slice exactly
    once, a wide access is aligned for x, cos and sin, the heads per thread
    leave at most a quarter of head slots idle, and each path appears only
    where it applies (rules of rope_partial_plan in include/rope_partial.h)."""
    for k in range(N_TABLE):
        c = fc.table_case(k)
        plan = host_plan(c)
        B, S, N, D = c.shape
        e = synth.ELEM_BYTES[c.dtype]
        L, st = c.sl.L, c.sl.start
        what = f"{c} -> path {plan.path} vec {plan.vec_bytes} U {plan.heads_per_thread} C {plan.chunks_per_row}"
        if plan.path == 0:
            assert L == 0 or B * S * N == 0, what
            continue
        U, C, vec = plan.heads_per_thread, plan.chunks_per_row, plan.vec_bytes
        assert U in (1, 2, 4, 8) and U <= max(N, 1), what
        slots = -(-N // U) * U
        assert U == 1 or (slots - N) * 4 <= slots, what
        assert plan.tasks == B * S * (-(-N // U)) * C, what
        half = c.mode == "half"
        if plan.path in (1, 3):
            # a wide access: whole chunks of the slice (of each half in half-split mode
            # with both halves in one thread), aligned everywhere
            covered = C * vec if (plan.path == 3 or not half) else 2 * C * vec
            assert covered == L * e, what
            assert (st * e) % vec == 0 and (D * e) % vec == 0, what
            assert (c.x_offset * e) % vec == 0 and (c.r_offset * e) % vec == 0, what
            rs = synth.r_shape_for(c.form, c.shape, L)
            if rs[0] * rs[1] * rs[2] > 1:  # several cos/sin rows, at a stride of L + pad
                assert ((L + c.r_pad) * e) % vec == 0, what
            assert plan.path != 3 or half, what
        elif plan.path == 2:
            assert C == L // 2 and vec == (e if half else 2 * e), what
        else:
            # a lane per aligned vector of x: the slice starts at element 1
            # of its vector, whose VE elements hold the first elements of
            # VE / 2 pairs, so a row of P pairs takes (P - 1) // (VE / 2) + 1
            # lanes
            assert plan.path == 4, what
            assert not half and st % 2 == 1, what
            assert vec in (16, 8), what
            assert (c.x_offset * e) % vec == 0 and (D * e) % vec == 0, what
            VE = vec // e
            assert st % VE == 1, what
            assert C == (L // 2 - 1) // (VE // 2) + 1, what

"""Pin checks for the oracle's forward and backward, as plain functions.

Each check raises AssertionError when the oracle disagrees with something
fixed independently of it: a hand-worked example, a closed form evaluated by
a library routine, an exact special case, an invariant of the mathematics,
or the brute-force Jacobian.  ``test_oracle_pins.py`` runs them against the
oracle; ``test_oracle_mutants.py`` runs them against deliberately broken
copies of the oracle to show that each plausible mistake is caught.  Every
check covers both rotary modes: interleave (pairs (2i, 2i+1)) and half
(pairs (i, i + L/2)).

Sources: "CANN ops-transformer inplace_partial_rotary_mul" (section
功能与计算公式 for the formula, the in-place write-back and the start == end
no-op; the kernel op chain in the same section; the backward's empty-tensor
no-op), and "ANE实战 RoPE位置编码在MIL中的纯ANE实现" (table recipe in 第一步,
rotate_half in 先搞懂RoPE, the inverse-rotation backward in 反向传播).
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
from oracle import rope_mil
from place_partial_rope_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DTYPES = ("fp32", "bf16", "fp16")
MODES = ("interleave", "half")
UNIT_ROUND = {"fp32": 2.0**-24, "bf16": 2.0**-8, "fp16": 2.0**-11}


def bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


def assert_bitwise(a, b, what=""):
    ba, bb = bits(np.ascontiguousarray(a)), bits(np.ascontiguousarray(b))
    bad = np.nonzero(ba.ravel() != bb.ravel())[0]
    assert bad.size == 0, f"{what}: {bad.size} lanes differ, first flat index {bad[:4]}"


def w(a, dtype):
    return oracle.widen(a, dtype).astype(np.float64)


def first(a, mode):
    """The first lane of every pair along the last axis."""
    return a[..., 0::2] if mode == "interleave" else a[..., : a.shape[-1] // 2]


def second(a, mode):
    """The second lane of every pair, aligned with first()."""
    return a[..., 1::2] if mode == "interleave" else a[..., a.shape[-1] // 2:]


def join(p, q, mode):
    """Inverse of (first, second): lanes p and q back in slice order."""
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.result_type(p, q))
    if mode == "interleave":
        out[..., 0::2], out[..., 1::2] = p, q
    else:
        h = p.shape[-1]
        out[..., :h], out[..., h:] = p, q
    return out


def swap(a, mode):
    return join(second(a, mode), first(a, mode), mode)


# --------------------------------------------------------------------------


def check_worked_example():
    for fname in ("interleave_worked_example.json", "half_split_worked_example.json"):
        with open(os.path.join(GOLDEN, fname)) as f:
            ex = json.load(f)
        mode = ex.get("mode", "interleave")
        shape, start, end = tuple(ex["shape"]), ex["start"], ex["end"]
        rs = tuple(ex["r_shape"])
        for dt in DTYPES:
            x = synth.to_storage(np.array(ex["x"], np.float64).reshape(shape), dt)
            g = synth.to_storage(np.array(ex["grad"], np.float64).reshape(shape), dt)
            c = synth.to_storage(np.array(ex["cos"], np.float64).reshape(rs), dt)
            s = synth.to_storage(np.array(ex["sin"], np.float64).reshape(rs), dt)
            want_f = synth.to_storage(np.array(ex["fwd"], np.float64).reshape(shape), dt)
            want_b = synth.to_storage(np.array(ex["bwd"], np.float64).reshape(shape), dt)
            for form in (oracle.GATHER_CHAIN, oracle.PAIR_ROTATION):
                assert_bitwise(oracle.fwd(x, c, s, dt, start, end, form, mode), want_f,
                               f"{mode} fwd {dt} {form}")
                assert_bitwise(oracle.bwd(g, c, s, dt, start, end, form, mode), want_b,
                               f"{mode} bwd {dt} {form}")
            assert_bitwise(rope_mil.fwd(x, c, s, dt, start, end, mode), want_f, f"{mode} mil fwd {dt}")
            assert_bitwise(rope_mil.bwd(g, c, s, dt, start, end, mode), want_b, f"{mode} mil bwd {dt}")


def check_formulations_agree():
    """The gather chain, the pair rotation and the array-level lowering give
    the same bits (forward and backward) on random shapes and broadcasts."""
    cases = [((2, 5, 3, 20), 2, 14, "BS1D"), ((1, 3, 4, 16), 3, 13, "BSND"),
             ((3, 1, 2, 12), 0, 12, "B11D"), ((2, 4, 1, 10), 4, 6, "111D"),
             ((2, 3, 5, 8), 0, 8, "1S1D")]
    for mode in MODES:
        for dt in DTYPES:
            for k, (shape, st, en, form) in enumerate(cases):
                x, c, s, g = synth.case(shape, st, en, dt, form, seed=10 + k)
                for fn_c, fn_m, inp in ((oracle.fwd, rope_mil.fwd, x), (oracle.bwd, rope_mil.bwd, g)):
                    a = fn_c(inp, c, s, dt, st, en, oracle.GATHER_CHAIN, mode)
                    b = fn_c(inp, c, s, dt, st, en, oracle.PAIR_ROTATION, mode)
                    m = fn_m(inp, c, s, dt, st, en, mode)
                    assert_bitwise(a, b, f"{mode} chain/pair {dt} {shape}")
                    assert_bitwise(a, m, f"{mode} chain/mil {dt} {shape}")


def check_complex_closed_form(formulation=oracle.GATHER_CHAIN):
    """With a table that repeats each pair's angle in both of its lanes, the
    forward is the complex product (x_m + i x_n)(c + i s) and the backward is
    (g_m + i g_n)(c - i s); numpy's complex128 multiply gives the exact value
    of both.  Bound: two product roundings and one sum rounding in fp32, then
    one rounding to the storage type."""
    shape, st, en = (2, 6, 3, 24), 4, 20
    for mode in MODES:
        for dt in DTYPES:
            x, c, s, g = synth.case(shape, st, en, dt, "BS1D", seed=3, table="rope", layout=mode)
            cf, sf = first(w(c, dt), mode), first(w(s, dt), mode)
            assert np.array_equal(cf, second(w(c, dt), mode))  # the table repeats each angle
            for direction, inp in ((oracle.FWD, x), (oracle.BWD, g)):
                out = oracle.rope(direction, inp, c, s, dt, st, en, formulation, mode)
                v = w(inp, dt)[..., st:en]
                vm, vn = first(v, mode), second(v, mode)
                z = (vm + 1j * vn) * (cf + 1j * (sf if direction == 0 else -sf))
                got = w(out, dt)[..., st:en]
                exact = join(z.real, z.imag, mode)
                mag = join(np.abs(vm * cf) + np.abs(vn * sf), np.abs(vn * cf) + np.abs(vm * sf), mode)
                tol = 2.0**-24 * 2.02 * mag + UNIT_ROUND[dt] * 1.01 * np.abs(exact) + 1e-30
                err = np.abs(got - exact)
                assert np.all(err <= tol), f"closed form {mode} {dt} dir {direction}: {err.max()}"


def check_special_cases(formulation=oracle.GATHER_CHAIN):
    """c=1, s=0 is the identity; c=0, s=1 is the exact quarter turn of each
    pair (a, b) -> (-b, a) forward and (a, b) -> (b, -a) backward; four
    quarter turns return the input bit for bit."""
    shape, st, en = (2, 3, 2, 16), 2, 14
    L = en - st
    for mode in MODES:
        for dt in DTYPES:
            x, _, _, _ = synth.case(shape, st, en, dt, "111D", seed=5)
            one = synth.to_storage(np.ones((1, 1, 1, L)), dt)
            zero = synth.to_storage(np.zeros((1, 1, 1, L)), dt)
            for fn in (oracle.fwd, oracle.bwd):
                assert_bitwise(fn(x, one, zero, dt, st, en, formulation, mode), x, f"identity {dt}")
            v = w(x, dt)[..., st:en]
            want = np.array(x, copy=True)
            want[..., st:en] = synth.to_storage(join(-second(v, mode), first(v, mode), mode), dt)
            assert_bitwise(oracle.fwd(x, zero, one, dt, st, en, formulation, mode), want,
                           f"quarter turn fwd {mode} {dt}")
            want[..., st:en] = synth.to_storage(join(second(v, mode), -first(v, mode), mode), dt)
            assert_bitwise(oracle.bwd(x, zero, one, dt, st, en, formulation, mode), want,
                           f"quarter turn bwd {mode} {dt}")
            y = x
            for _ in range(4):
                y = oracle.fwd(y, zero, one, dt, st, en, formulation, mode)
            assert_bitwise(y, x, f"four quarter turns {mode} {dt}")


def check_invariants(formulation=oracle.GATHER_CHAIN):
    """Pair norms are kept; bwd(fwd(x)) returns x within 1e-6 of each pair's
    norm in fp32 with a cos/sin table; bytes outside [start, end) never
    change; start == end and an empty tensor are no-ops."""
    shape, st, en = (2, 8, 4, 40), 6, 38
    for mode in MODES:
        x, c, s, _ = synth.case(shape, st, en, "fp32", "BS1D", seed=8, table="rope", layout=mode)
        y = oracle.fwd(x, c, s, "fp32", st, en, formulation, mode)
        xs, ys = x[..., st:en].astype(np.float64), y[..., st:en].astype(np.float64)
        n_in = first(xs, mode) ** 2 + second(xs, mode) ** 2
        n_out = first(ys, mode) ** 2 + second(ys, mode) ** 2
        cn = first(c.astype(np.float64), mode) ** 2 + first(s.astype(np.float64), mode) ** 2
        assert np.allclose(n_out, n_in * cn, rtol=4e-7, atol=1e-30), f"pair norm {mode}"
        back = oracle.bwd(y, c, s, "fp32", st, en, formulation, mode)
        # a rotation mixes the two lanes of a pair, so a small lane carries
        # its partner's rounding: measure against the pair's norm
        err = np.abs(back[..., st:en].astype(np.float64) - xs)
        norm = np.sqrt(n_in)
        rel = err / join(norm, norm, mode)
        assert rel.max() <= 1e-6, f"bwd(fwd(x)) {mode}: {rel.max()}"
        assert_bitwise(back[..., :st], x[..., :st], "bwd(fwd) left of slice")
        for dt in DTYPES:
            xd, cd, sd, gd = synth.case(shape, st, en, dt, "BSND", seed=9)
            for fn, inp in ((oracle.fwd, xd), (oracle.bwd, gd)):
                out = fn(inp, cd, sd, dt, st, en, formulation, mode)
                assert_bitwise(out[..., :st], inp[..., :st], f"left of slice {dt}")
                assert_bitwise(out[..., en:], inp[..., en:], f"right of slice {dt}")
                assert not np.array_equal(bits(out[..., st:en]), bits(inp[..., st:en]))
            empty_r = np.zeros((1, 1, 1, 0), xd.dtype)
            for fn in (oracle.fwd, oracle.bwd):
                assert_bitwise(fn(xd, empty_r, empty_r, dt, 10, 10, formulation, mode), xd, "start==end")
                e = np.zeros((0, 3, 4, 40), xd.dtype)
                assert fn(e, cd[:1], sd[:1], dt, st, en, formulation, mode).shape == e.shape


def check_backward_is_transpose(formulation=oracle.GATHER_CHAIN):
    """Brute force: column k of the forward's Jacobian is fwd(e_k) and row m of
    the backward's is bwd(e_m); with unit inputs every entry is a single table
    value (exact), so bwd must be the forward's transpose bit for bit.  The
    table is random and per head, so every lane index is pinned; each pair's
    2x2 block must be [[c_m, -s_m], [s_n, c_n]]."""
    shape, st, en = (1, 2, 2, 8), 2, 8
    n = int(np.prod(shape))
    L = en - st
    for mode in MODES:
        for dt in DTYPES:
            _, c, s, _ = synth.case(shape, st, en, dt, "BSND", seed=21)
            one = synth.to_storage(np.ones(1), dt)[0]
            Jf = np.zeros((n, n))
            Jb = np.zeros((n, n))
            for k in range(n):
                e = np.zeros(n, c.dtype)
                e[k] = one
                e = e.reshape(shape)
                Jf[:, k] = w(oracle.fwd(e, c, s, dt, st, en, formulation, mode), dt).ravel()
                Jb[:, k] = w(oracle.bwd(e, c, s, dt, st, en, formulation, mode), dt).ravel()
            assert np.array_equal(Jb, Jf.T), f"bwd is not the transpose of fwd ({mode} {dt})"
            cw, sw = w(c, dt), w(s, dt)
            pairs = ([(2 * i, 2 * i + 1) for i in range(L // 2)] if mode == "interleave"
                     else [(i, i + L // 2) for i in range(L // 2)])
            for b_ in range(shape[0]):
                for s_ in range(shape[1]):
                    for h in range(shape[2]):
                        base = ((b_ * shape[1] + s_) * shape[2] + h) * shape[3]
                        for m, q in pairs:
                            p_, r_ = base + st + m, base + st + q
                            blk = Jf[np.ix_([p_, r_], [p_, r_])]
                            want = [[cw[b_, s_, h, m], -sw[b_, s_, h, m]],
                                    [sw[b_, s_, h, q], cw[b_, s_, h, q]]]
                            assert np.array_equal(blk, np.array(want)), f"pair block {mode} {dt}"
            outside = [i for i in range(n) if not st <= i % shape[3] < en]
            assert np.array_equal(Jf[np.ix_(outside, outside)], np.eye(len(outside)))


def check_adjoint_identity(formulation=oracle.GATHER_CHAIN):
    """<fwd(x), g> = <x, bwd(g)> for random, non-duplicated tables, within the
    rounding of the two products and the sum of each lane."""
    shape, st, en = (3, 7, 5, 36), 2, 30
    for mode in MODES:
        for dt in DTYPES:
            x, c, s, g = synth.case(shape, st, en, dt, "B1ND", seed=31)
            fx = w(oracle.fwd(x, c, s, dt, st, en, formulation, mode), dt)[..., st:en]
            bg = w(oracle.bwd(g, c, s, dt, st, en, formulation, mode), dt)[..., st:en]
            xv, gv = w(x, dt)[..., st:en], w(g, dt)[..., st:en]
            lhs, rhs = np.sum(fx * gv), np.sum(xv * bg)
            cw = np.abs(np.broadcast_to(w(c, dt), xv.shape))
            sw = np.abs(np.broadcast_to(w(s, dt), xv.shape))
            # per-lane magnitude bounds of the rounded forward and backward lanes
            mag_f = np.abs(xv) * cw + swap(np.abs(xv), mode) * sw
            mag_b = np.abs(gv) * cw + swap(np.abs(gv) * sw, mode)
            scale = np.sum(mag_f * np.abs(gv)) + np.sum(np.abs(xv) * mag_b)
            tol = (2 * 2.0**-24 + UNIT_ROUND[dt]) * 1.05 * scale
            assert abs(lhs - rhs) <= tol, f"adjoint {mode} {dt}: {lhs} vs {rhs} (tol {tol})"


def check_conversions():
    """The storage roundings against library conversions on every tie and
    its neighbours (a smaller version of test_oracle_conversions.py)."""
    import torch
    hi = np.arange(0, 2**16, 7, dtype=np.uint32) << 16
    vals = np.concatenate([hi | np.uint32(0x8000 + d) for d in (-1, 0, 1)]).view(np.float32)
    vals = vals[np.isfinite(vals)]
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f32_to_bf16(vals), ref), "bf16 rounding"
    h = np.arange(0, 0x7C00, 3, dtype=np.uint16)
    mid = ((h.view(np.float16).astype(np.float64) +
            (h + 1).view(np.float16).astype(np.float64)) / 2).astype(np.float32)
    mb = mid.view(np.uint32).astype(np.int64)
    cand = np.concatenate([(mb + d).astype(np.uint32) for d in (-1, 0, 1)]).view(np.float32)
    cand = cand[np.isfinite(cand)]
    with np.errstate(over="ignore"):
        ref16 = cand.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f32_to_f16(cand), ref16), "fp16 rounding"


ALL_CHECKS = [check_worked_example, check_formulations_agree, check_complex_closed_form,
              check_special_cases, check_invariants, check_backward_is_transpose,
              check_adjoint_identity, check_conversions]

"""The odd-start kernel's lane arithmetic, emulated on the CPU.

rope_partial_odd_kernel gives each lane one aligned V-byte vector of x when
the slice starts at element 1 of such a vector.  Lane j of a row rotates the
pairs whose first element lies in its vector, takes the last pair's second
element from the next lane (a shuffle) or, where no next lane of the row is
in its warp, loads that word itself; it receives its own element 0 from the
previous lane's last result (a shuffle) and stores the elements of its
vector that belong to the slice, plus element 0 of the next vector when no
lane of its warp will.  This test replays that arithmetic lane by lane:
whole warps of 32 consecutive work items, every lane's loads (all heads)
before any of its stores, dead lanes past the end of the work, and warps
taken in both orders.  It asserts that every read of x stays inside its row
and every read of cos/sin inside its table row, that every write lands in
the slice and each slice element is written exactly once, and that the
result equals the oracle bit for bit (a race between warps would make the
two orders disagree with it).  Host only: no GPU, no CUDA.
"""
import numpy as np
import pytest

import oracle
from place_partial_rope_gb300 import synth

E = {"bf16": 2, "fp16": 2, "fp32": 4}


def rotate(direction, x0, x1, c0, c1, s0, s1):
    """One pair in fp32, each product and sum one rounding (the kernel's
    rotate_pair)."""
    f = np.float32
    if direction == "fwd":
        return f(f(x0 * c0) - f(x1 * s0)), f(f(x1 * c1) + f(x0 * s1))
    return f(f(x0 * c0) + f(x1 * s1)), f(f(x1 * c1) - f(x0 * s0))


def emulate(direction, x, c, s, dtype, start, end, V, U, reverse):
    """x: (B, S, N, D) storage values; c, s: broadcastable (Br, Sr, Nr, L).
    Returns the emulated result (storage values) and the write count."""
    B, S, N, D = x.shape
    e = E[dtype]
    VE = V // e                      # elements per vector
    PV = VE // 2                     # pair slots per lane
    L = end - start
    P = L // 2
    assert start % VE == 1
    C = (P - 1) // PV + 1            # lanes per row
    H = -(-N // U)                   # head groups
    tasks = B * S * H * C
    mem = x.reshape(-1).copy()
    wide = oracle.widen(mem, dtype).astype(np.float32)  # fp32 view of the inputs
    cw = oracle.widen(c, dtype).astype(np.float32)
    sw_ = oracle.widen(s, dtype).astype(np.float32)
    written = set()

    def table(tab, b, si, n, q):
        Br, Sr, Nr, Lr = tab.shape
        assert 0 <= q < Lr, ("cos/sin read outside its row", q)
        return tab[b if Br > 1 else 0, si if Sr > 1 else 0, n if Nr > 1 else 0, q]

    def read(row0, col):
        assert 0 <= col < D, ("x read outside its row", col)
        return wide[row0 + col]

    order = list(range(0, tasks, 32))
    if reverse:
        order.reverse()
    for base in order:
        lanes = {}
        for lane in range(32):
            t = base + lane
            if t >= tasks:
                continue  # dead: reads and writes nothing
            j, rest = t % C, t // C
            hg, tok = rest % H, rest // H
            w0 = j * PV
            m_hi = min(PV, P - w0)
            ends_next = m_hi == PV
            lanes[lane] = dict(
                j=j, b=tok // S, s=tok % S, tok=tok, hg=hg, w0=w0, m_hi=m_hi,
                prev_here=j > 0 and lane != 0,
                store_next=ends_next and (j + 1 == C or lane == 31),
                vs=start - 1 + j * VE)  # the vector's element 0, in the row
        # the kernel loads every head of a lane before it stores any
        for q in lanes.values():
            q["heads"] = [i for i in range(U) if q["hg"] * U + i < N]
            q["x"], q["nx"] = {}, {}
            for i in q["heads"]:
                row0 = (q["tok"] * N + q["hg"] * U + i) * D
                q["x"][i] = [read(row0, q["vs"] + k) for k in range(VE)]
                if q["store_next"]:  # the next vector's first word
                    word = [read(row0, q["vs"] + VE + k) for k in range(4 // e)]
                    q["nx"][i] = word[0]
        for i in range(U):
            y = {}
            for lane, q in lanes.items():
                if i not in q["heads"]:
                    continue
                n = q["hg"] * U + i
                xv = q["x"][i]
                nxt = lanes.get(lane + 1)  # shuffle down: the next lane's element 0
                down = nxt["x"][i][0] if (nxt is not None and i in nxt["x"]) else np.float32(0)
                after = q["nx"][i] if q["store_next"] else down
                pairs = []
                for m in range(PV):
                    if m < q["m_hi"]:
                        p = q["w0"] + m
                        x0 = xv[2 * m + 1]
                        x1 = xv[2 * m + 2] if 2 * m + 2 < VE else after
                        c0, c1 = table(cw, q["b"], q["s"], n, 2 * p), table(cw, q["b"], q["s"], n, 2 * p + 1)
                        s0, s1 = table(sw_, q["b"], q["s"], n, 2 * p), table(sw_, q["b"], q["s"], n, 2 * p + 1)
                        pairs.append(rotate(direction, x0, x1, c0, c1, s0, s1))
                    else:
                        pairs.append((np.float32(0), np.float32(0)))  # not stored
                y[lane] = pairs
            for lane, q in lanes.items():
                if i not in q["heads"]:
                    continue
                row0 = (q["tok"] * N + q["hg"] * U + i) * D
                prv = lanes.get(lane - 1)  # shuffle up: the previous lane's last second result
                prev = y[lane - 1][PV - 1][1] if (prv is not None and lane - 1 in y) else np.float32(0)
                vals = [prev] + [v for pair in y[lane] for v in pair]  # element k of the vector
                lo = 0 if q["prev_here"] else 1
                hi = min(2 * q["m_hi"] + 1, VE)
                ks = list(range(lo, hi)) + ([VE] if q["store_next"] else [])
                for k in ks:
                    col = q["vs"] + k
                    assert start <= col < end, ("write outside the slice", col)
                    assert (row0, col) not in written, ("element written twice", row0, col)
                    written.add((row0, col))
                    mem[row0 + col] = oracle.narrow(np.array([vals[k]], np.float32), dtype)[0]
    return mem.reshape(x.shape), len(written)


def cases():
    rng = np.random.default_rng(7)
    out = []
    forms = ["BSND", "1S1D", "BS1D", "B11D", "111D", "11ND"]
    for dtype in ("bf16", "fp16", "fp32"):
        e = E[dtype]
        for V in (16, 8):
            VE = V // e
            for D in (8, 16, 24, 40, 64, 136):
                if (D * e) % V:
                    continue
                for start in range(1, D, VE):
                    for L in sorted({2, 4, 6, 14, 16, 30, 32, 62, 64, D - start - 1}):
                        if L > 0 and L % 2 == 0 and start + L <= D:
                            out.append((dtype, V, D, start, start + L))
    rng.shuffle(out)
    sel = []
    for k, (dtype, V, D, start, end) in enumerate(out[:120]):
        N = int(rng.integers(1, 7))
        U = int(rng.choice([1, 2, 4, 8]))
        B, S = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        sel.append((dtype, V, (B, S, N, D), start, end, U, forms[k % 6], k))
    return sel


@pytest.mark.parametrize("dtype,V,shape,start,end,U,form,seed", cases())
def test_odd_lanes_match_the_oracle(dtype, V, shape, start, end, U, form, seed):
    x, c, s, g = synth.case(shape, start, end, dtype, form, seed=seed)
    B, S, N, D = shape
    for direction, inp in (("fwd", x), ("bwd", g)):
        want = (oracle.fwd if direction == "fwd" else oracle.bwd)(inp, c, s, dtype, start, end)
        view = np.uint32 if dtype == "fp32" else np.uint16
        for reverse in (False, True):
            got, nwritten = emulate(direction, inp, c, s, dtype, start, end, V, U, reverse)
            assert nwritten == B * S * N * (end - start)
            assert np.array_equal(got.view(view), want.view(view)), (direction, reverse)


def test_cases_reach_rows_that_straddle_warps_and_every_width():
    """The draws include rows whose lanes do not divide 32 (a row then spans
    two warps: the last lane of a warp loads the next vector's word and
    stores the straddling element itself) and every (element size, vector
    width) pair."""
    seen, straddle = set(), 0
    for dtype, V, shape, start, end, U, form, seed in cases():
        e = E[dtype]
        PV = V // e // 2
        C = ((end - start) // 2 - 1) // PV + 1
        seen.add((e, V))
        straddle += 32 % C != 0
    assert seen == {(2, 16), (2, 8), (4, 16), (4, 8)}
    assert straddle >= 10

// rope_host.cpp -- the C ABI entry points of include/rope_partial.h.
//
// Everything here is host logic: argument validation (the constraint list of
// "CANN ops-transformer inplace_partial_rotary_mul", section 约束说明),
// broadcast-stride resolution for cos/sin, the empty-call rule (section
// 功能与计算公式: start == end leaves x unchanged; the backward accepts empty
// tensors), the choice of kernel path and access width, grid sizing, and the
// split of very large calls into launches whose flat work index fits 32 bits.
// No CUDA call is made before the arguments have been validated, and none
// at all for a rejected or empty call.
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "rope_internal.h"

namespace rope {
namespace {

thread_local char g_msg[512] = "";

rope_status_t fail(rope_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

// Prefix the current message (copied first: vsnprintf must not read the
// buffer it writes).
rope_status_t fail_prefixed(rope_status_t st, const char* prefix) {
    char tmp[sizeof(g_msg)];
    snprintf(tmp, sizeof(tmp), "%s", g_msg);
    return fail(st, "%s: %s", prefix, tmp);
}

int elem_bytes(int dtype) { return dtype == ROPE_FP32 ? 4 : 2; }

struct Resolved {
    int e = 0;
    int64_t L = 0;
    bool empty = false;
    int64_t rb[2][3] = {{0, 0, 0}, {0, 0, 0}};  // byte strides (b, s, n); 0 on broadcast dims
};

bool mul_overflows(int64_t a, int64_t b) { return a != 0 && b > INT64_MAX / a; }

rope_status_t check(const void* x, const void* r1, const void* r2, int dtype, int64_t B,
                    int64_t S, int64_t N, int64_t D, const int64_t* r1_shape,
                    const int64_t* r1_stride, const int64_t* r2_shape, const int64_t* r2_stride,
                    int64_t start, int64_t end, Resolved* out) {
    if (dtype != ROPE_BF16 && dtype != ROPE_FP16 && dtype != ROPE_FP32)
        return fail(ROPE_ERR_INVALID, "dtype %d is not bf16 (0), fp16 (1) or fp32 (2)", dtype);
    if (B < 0 || S < 0 || N < 0 || D < 0)
        return fail(ROPE_ERR_INVALID, "negative size: B=%lld S=%lld N=%lld D=%lld", (long long)B,
                    (long long)S, (long long)N, (long long)D);
    if (D % 2 != 0) return fail(ROPE_ERR_INVALID, "head dim D=%lld must be even", (long long)D);
    if (D > 1024) return fail(ROPE_ERR_INVALID, "head dim D=%lld exceeds 1024", (long long)D);
    if (start < 0 || end < start || end > D)
        return fail(ROPE_ERR_INVALID, "partial slice [%lld, %lld) must satisfy 0 <= start <= end <= D=%lld",
                    (long long)start, (long long)end, (long long)D);
    const int64_t L = end - start;
    if (L % 2 != 0)
        return fail(ROPE_ERR_INVALID, "slice length end - start = %lld must be even", (long long)L);

    const bool empty = L == 0 || B == 0 || S == 0 || N == 0 || D == 0;
    const int64_t xdim[3] = {B, S, N};
    const int64_t* shapes[2] = {r1_shape, r2_shape};
    const int64_t* strides[2] = {r1_stride, r2_stride};
    for (int r = 0; r < 2; ++r) {
        if (!shapes[r]) {
            if (empty) continue;
            return fail(ROPE_ERR_NULLPTR, "r%d_shape is null", r + 1);
        }
        for (int k = 0; k < 3; ++k)
            if (!(shapes[r][k] == 1 || shapes[r][k] == xdim[k]))
                return fail(ROPE_ERR_INVALID, "r%d dim %d is %lld; it must be 1 or %lld to broadcast",
                            r + 1, k, (long long)shapes[r][k], (long long)xdim[k]);
        if (shapes[r][3] != L)
            return fail(ROPE_ERR_INVALID, "r%d last dim is %lld; it must equal end - start = %lld",
                        r + 1, (long long)shapes[r][3], (long long)L);
    }
    out->L = L;
    out->e = elem_bytes(dtype);
    if (empty) {
        out->empty = true;
        return ROPE_OK;
    }

    if (!x) return fail(ROPE_ERR_NULLPTR, "x is null");
    if (!r1) return fail(ROPE_ERR_NULLPTR, "r1 (cos) is null");
    if (!r2) return fail(ROPE_ERR_NULLPTR, "r2 (sin) is null");
    const int e = out->e;
    int64_t total = B;
    if (mul_overflows(total, S) || mul_overflows(total * S, N) || mul_overflows(total * S * N, D) ||
        mul_overflows(total * S * N * D, e))
        return fail(ROPE_ERR_INVALID, "x of %lld x %lld x %lld x %lld elements overflows 64-bit bytes",
                    (long long)B, (long long)S, (long long)N, (long long)D);
    for (int r = 0; r < 2; ++r) {
        if (!strides[r]) return fail(ROPE_ERR_NULLPTR, "r%d_stride is null", r + 1);
        if (L > 1 && strides[r][3] != 1)
            return fail(ROPE_ERR_INVALID, "r%d last-dim stride is %lld; it must be 1 (contiguous)",
                        r + 1, (long long)strides[r][3]);
        for (int k = 0; k < 3; ++k) {
            if (shapes[r][k] == 1) {
                out->rb[r][k] = 0;
                continue;
            }
            if (strides[r][k] < 0)
                return fail(ROPE_ERR_INVALID, "r%d stride %d is negative (%lld)", r + 1, k,
                            (long long)strides[r][k]);
            if (mul_overflows(strides[r][k], shapes[r][k] * e))
                return fail(ROPE_ERR_INVALID, "r%d stride %d overflows", r + 1, k);
            out->rb[r][k] = strides[r][k] * e;
        }
    }
    if (reinterpret_cast<uintptr_t>(x) % e || reinterpret_cast<uintptr_t>(r1) % e ||
        reinterpret_cast<uintptr_t>(r2) % e)
        return fail(ROPE_ERR_INVALID, "x, r1 and r2 must be aligned to their %d-byte elements", e);
    return ROPE_OK;
}

// Heads per thread: the largest power of two U <= min(cap, N) whose
// ceil(N / U) * U head slots leave at most a quarter idle.  An idle slot
// costs issue slots, not memory traffic, so a larger U (more accesses in
// flight, cos/sin reused more) wins over a perfect fit.
//
// The cap comes from back-to-back timings on GB300 of every access kind
// (U = 1, 2, 4, 8, and both grids, on the workloads' shapes and on other
// slices of them).  fp32 rows want about 32 bytes of x per thread: 8-byte
// accesses of the large shape's slice at byte 136 ran 99.5 us at U = 4
// against 110.8 us at 2 and 100.4 us at 8 (the positions call: 97.1 us);
// 16-byte accesses ran 82.7 us at U = 2 against 83.2 us at 4 ([32, 96))
// and 159.7 against 160.0 us (the whole 512-byte row).  16-bit rows:
// 16-byte accesses want 4 (gqa 42.0 us; flat from 2 to 8 on 256-byte rows,
// best at 4 on 384-byte rows), 8-byte ones 2 (55.5 us against 57.7 at 4)
// and 4-byte ones 4 (57.5 us against 71.9 at 2).  The half-split kernel that
// takes its partner from another lane wants more in flight (8-byte accesses
// 56.5 us at U = 4 against 57.4 at 2; 4-byte ones 57.4 us at 8 against 59.6
// at 4).  The half-split kernel with both halves in one thread (table call,
// on the full grid): fp32 2 on 16- and 8-byte accesses ([0, 96) 118.9 us
// against 148.9 at 1 and 119.5 at 4; [2, 98) 133.0 against 153.3 at 1) and
// 8 on 4-byte ones ([1, 97) 152.2 against 154.7 at 4); 16-bit 4 on 16-byte
// accesses (gqa shape [0, 96) 61.3 us against 69.2 at 1; [0, 48) 38.7
// against 37.8 at 1 and 45.7 at 2) and 8 on 8- and 4-byte ones ([4, 52)
// 36.6 against 38.8 at 2; [2, 50) 39.3 against 41.6 at 2).  The positions
// call computes each thread's angles once for all its heads, so it wants
// more of them: fp32 4 on 16- and 8-byte accesses ([32, 96) 78.5 us
// against 88.3 at 2), 2 with both halves in one thread on 16-byte ones
// ([0, 96) 115.8 against 134.0 at 1); 16-bit 4 on 8-byte accesses ([4, 68)
// 54.7 against 58.6 at 2) and 8 on 4-byte ones ([2, 66) 54.7 against 59.5
// at 4), 2 with both halves in one thread (gqa 44.8 us against 47.4 at 4).
// The element path is best at 8 (4 with both halves in one thread).
// Short 16-bit slices of 16-byte accesses want fewer heads: on the gqa shape
// [0, 16) (2 accesses per row) ran 23.8 us at U = 1 against 32.7 at 4
// (half-split 24.8 against 31.2), and 4-access slices 25.2 us at U = 2
// against 27.7 at 4 ([0, 32), [32, 64), [64, 96); [16, 48) 32.7 against
// 35.7); from 6 accesses on 4 stays best ([0, 48) 36.4 us), and so it does
// for half-split rows of 4 accesses ([0, 32) 27.2 against 28.2 at 2).  (On
// the MLA-decode shape, whose short slices stay in L2 back to back, U = 4
// ran those 8 % faster there and level after an L2 flush.)
// The odd-start kernel (a lane per aligned vector of x, vec bytes): 4 heads
// per thread on 16-byte vectors (the most that kernel instance allows), 8
// on 8-byte ones.  Back to back on GB300: GQA [9, 73) 16-byte 56.9 us (U
// = 4) against 60.7 (2); [5, 69) 8-byte 58.3 (8) against 64.8 (4); large
// fp32 [1, 65) 16-byte 98.8 (4) against 113.8 (2), [3, 67) 8-byte 102.9
// (8) against 118.0 (4).
int odd_heads_cap(int e, int vec) {
    (void)e;
    return vec == 16 ? 4 : 8;
}

int heads_cap(int e, int vec, int path, bool pair, bool lanes, bool pos, int chunks) {
    if (path == kScalarPair) return pair ? 4 : 8;
    if (path == kOddPair) return odd_heads_cap(e, vec);
    if (e == 4) {
        if (pair) return vec == 4 ? (pos ? 4 : 8) : 2;
        if (pos) return 4;
        return vec >= 32 ? 1 : 32 / vec;  // about 32 bytes of x per thread
    }
    if (pair) return pos ? 2 : (vec == 16 ? 4 : 8);
    // 16-byte accesses of a short 16-bit row slice: one head per thread for
    // 2 accesses per row (interleave or half-split lanes), two for 4
    // (interleave)
    if (vec == 16 && chunks <= 2) return 1;
    if (vec == 16 && chunks <= 4 && !lanes) return 2;
    if (lanes) return vec == 16 ? 4 : (vec == 8 ? 4 : 8);
    if (pos) return vec == 4 ? 8 : 4;
    return vec == 8 ? 2 : 4;
}

int choose_heads_per_thread(int64_t N, int cap) {
    for (int u = cap; u > 1; u /= 2) {
        if (u > N) continue;
        const int64_t slots = ((N + u - 1) / u) * u;
        if ((slots - N) * 4 <= slots) return u;
    }
    return 1;
}

// One tensor whose slice a launch rotates: the single call has one, the
// fused query + key call two (heads of the second follow the first's).
struct Seg {
    void* x;
    int64_t N, D, start;
};

rope_status_t make_plan(int dir, int mode, int dtype, const Seg* seg, int nseg, const void* r1,
                        const void* r2, const Resolved& R, Plan* P, bool host = false,
                        bool pos = false) {
    const int e = R.e;
    const bool half = mode == kHalf;
    // interleave: an access holds whole pairs; half-split: an access holds
    // lanes of the first half and its partner access lies L/2 lanes on
    const int64_t Lb = half ? (R.L / 2) * e : R.L * e;
    const uintptr_t p1 = reinterpret_cast<uintptr_t>(r1), p2 = reinterpret_cast<uintptr_t>(r2);
    int64_t N = 0;
    for (int i = 0; i < nseg; ++i) N += seg[i].N;
    int vec = 0;
    for (int v = 16; v >= 4; v /= 2) {
        if (!half && v < 2 * e) break;  // an access must hold whole pairs
        bool ok = Lb % v == 0 && p1 % v == 0 && p2 % v == 0;
        for (int i = 0; i < nseg; ++i)
            ok = ok && (seg[i].start * e) % v == 0 && (seg[i].D * e) % v == 0 &&
                 reinterpret_cast<uintptr_t>(seg[i].x) % v == 0;
        for (int r = 0; r < 2; ++r)
            for (int k = 0; k < 3; ++k) ok = ok && R.rb[r][k] % v == 0;
        if (ok) {
            vec = v;
            break;
        }
    }
    P->dtype = dtype;
    P->dir = dir;
    P->two = nseg == 2;
    P->half = half;
    // Interleave with an odd start (one tensor, table call): every pair
    // straddles two aligned accesses.  A lane per aligned V-byte vector of x,
    // V the wider of 16 and 8 bytes that divides x's address and its row
    // pitch and puts the start at element 1 of a vector (start = 1 modulo
    // V / e; at 8 bytes that is any odd start for fp32, and starts = 1 or 5
    // modulo 8 for 16-bit types).  cos/sin are loaded a pair at a time (a
    // 4-byte word per 16-bit pair, two per fp32 pair, so their rows must be
    // 4-byte aligned), or one V-byte access per lane when their rows are
    // V-aligned.  A lane's vector holds VE = V / e elements and the first
    // elements of PV = VE / 2 pairs, so a row takes (P - 1) / PV + 1 lanes for
    // its P pairs.  Back to back on GB300 against the element path (device
    // time, steady): GQA [1, 65) 57.0 against 73.4 us, [1, 63) 52.1 against
    // 58.0, [5, 69) at 8 bytes 58.3 against 73.3, [13, 71) 67.4 against 84.4,
    // x 8 bytes off 16 at [1, 65) 58.2 against 73.3; the MLA-decode query's
    // [1, 65) 31.5 against 43.1; large fp32 [1, 65) 98.7 against 108.0 and, at
    // 8 bytes, [3, 67) 102.8 against 108.2.  Other odd starts (16-bit starts
    // = 3 modulo 4, rows only 4-byte aligned) run the element path.
    const int64_t pairs = R.L / 2;
    int odd_v = 0;
    if (!vec && !half && !pos && nseg == 1 && (seg[0].start & 1)) {
        bool r4 = p1 % 4 == 0 && p2 % 4 == 0;
        for (int r = 0; r < 2; ++r)
            for (int k = 0; k < 3; ++k) r4 = r4 && R.rb[r][k] % 4 == 0;
        const uintptr_t px = reinterpret_cast<uintptr_t>(seg[0].x);
        const int64_t row = seg[0].D * e;
        // the widest vector that x's address and row pitch allow and that
        // puts the start at element 1 of a vector
        for (int v = 16; r4 && v >= 8; v /= 2)
            if (px % v == 0 && row % v == 0 && seg[0].start % (v / e) == 1) {
                odd_v = v;
                break;
            }
    }
    P->odd_wide = false;
    if (vec) {
        P->path = kVector;
        P->vec = vec;
        P->C = static_cast<int>(Lb / vec);
    } else if (odd_v) {
        P->path = kOddPair;
        P->vec = odd_v;
        const int PV = odd_v / e / 2;
        P->C = static_cast<int>((pairs - 1) / PV + 1);
        bool wide = p1 % odd_v == 0 && p2 % odd_v == 0;
        for (int r = 0; r < 2; ++r)
            for (int k = 0; k < 3; ++k) wide = wide && R.rb[r][k] % odd_v == 0;
        P->odd_wide = wide;
    } else if (half) {
        P->path = kScalarPair;  // a 16-bit slice not aligned for 4-byte accesses
        P->vec = e;
        P->C = static_cast<int>(R.L / 2);
    } else {
        P->path = kScalarPair;  // odd start, or a row not aligned for wide accesses
        P->vec = 2 * e;
        P->C = static_cast<int>(R.L / 2);
    }
    P->pos = pos;
    // Half-split rows of 2..32 accesses (a power of two) fit one warp: each
    // thread then takes one access and its partner's comes by shuffle.  Back
    // to back this ran the large fp32 shape in 102.9 us against 104.5-105.1
    // us with both halves in one thread (the interleave kernel: 103.0 us),
    // and gqa in 43.2 us against 44.6 us (interleave: 42.0 us); after an L2
    // flush the two are level (gqa 40-41 us, large fp32 100-102 us).  The
    // positions call keeps both halves in one thread: there each lane would
    // compute its partner's angles again, and the large fp32 shape ran 105.0
    // us that way against 103.9 us (gqa level at 47.3 against 47.8 us).
    const int64_t C_row = 2 * int64_t(P->C);
    P->lanes = half && !pos && P->path == kVector && C_row <= 32 && (C_row & (C_row - 1)) == 0;
    if (P->lanes) P->C = static_cast<int>(C_row);
    P->r_head = R.rb[0][2] != 0 || R.rb[1][2] != 0;
    // Host buffers (the *_host calls) are read across the host link, where
    // one head per thread ran fastest: gqa 0.81 ms against 0.87 ms with 4
    // (1.05 ms on the full grid), mla_decode_q 0.42 against 0.45 ms; the
    // large fp32 shape 2.18 ms against 2.26-2.30 ms with 2 or 4.
    const bool pair = half && !P->lanes;
    P->U = choose_heads_per_thread(seg[0].N,
                                   host ? 1 : heads_cap(e, P->vec, P->path, pair, P->lanes, pos, P->C));
    // Grid: a grid of one block per 256 work items, whose blocks the
    // hardware replaces as they finish, ran faster than a resident grid whose
    // threads stride over the work (the large fp32 shape 99.5 against 103.2
    // us, its positions call 97.1 against 103.9 us, [32, 96) 82.7 against
    // 86.9 us; gqa 42.0 against 44.7 us; the 16-bit element path in
    // half-split mode 75.8 against 83.8 us; the half-split kernel with both
    // halves in one thread, [0, 96) fp32 118.9 against 155.5 us at U = 2,
    // gqa shape [0, 96) 61.3 against 68.4 us at U = 4; the fused query + key
    // call, whose work index sweeps the query, then the key, 47.3 against
    // 51.2 us cold on a GQA pair).  The exception ran faster on the resident
    // grid: 16-bit rows read over the host link (mla_decode_q 422 against
    // 441 us; gqa level at 815-819 us, while the large fp32 shape there ran
    // 2184 against 2291 us on the full grid).
    P->full_grid = host ? (e == 4 && nseg == 1) : true;
    // head groups of each tensor (the fused call sweeps the first tensor's
    // items, then the second's)
    const int64_t H = (seg[0].N + P->U - 1) / P->U;
    const int64_t H2 = nseg == 2 ? (seg[1].N + P->U - 1) / P->U : 0;
    if ((H + H2) * P->C > int64_t(kMaxPieceTasks))
        return fail(ROPE_ERR_INVALID, "N=%lld heads with a %lld-lane slice exceed the per-token work "
                    "limit of 2^31 accesses", (long long)N, (long long)R.L);
    P->H = static_cast<int>(H);
    P->H2 = static_cast<int>(H2);
    return ROPE_OK;
}

KernelArgs base_args(const Plan& P, const Seg* seg, int nseg, const void* r1, const void* r2,
                     const Resolved& R) {
    KernelArgs k{};
    k.x = static_cast<char*>(seg[0].x) + seg[0].start * R.e;
    if (P.path == kOddPair) {
        // the odd-start kernel addresses whole vectors from the one that
        // holds element start (at its element 1)
        k.x -= R.e;
        k.pairs = static_cast<int32_t>(R.L / 2);
        k.odd_wide = P.odd_wide ? 1 : 0;
    }
    k.row_bytes = seg[0].D * R.e;
    k.tok_bytes = seg[0].N * seg[0].D * R.e;
    k.N1 = static_cast<int32_t>(seg[0].N);
    k.N = k.N1;
    if (nseg == 2) {
        k.x2 = static_cast<char*>(seg[1].x) + seg[1].start * R.e;
        k.row_bytes2 = seg[1].D * R.e;
        k.tok_bytes2 = seg[1].N * seg[1].D * R.e;
        k.N += static_cast<int32_t>(seg[1].N);
    }
    k.r1 = static_cast<const char*>(r1);
    k.r2 = static_cast<const char*>(r2);
    k.r1_b = R.rb[0][0];
    k.r1_s = R.rb[0][1];
    k.r1_n = R.rb[0][2];
    k.r2_b = R.rb[1][0];
    k.r2_s = R.rb[1][1];
    k.r2_n = R.rb[1][2];
    k.H = P.H;
    k.half_off = P.half ? (R.L / 2) * R.e : 0;
    k.divC = FastDiv::make(static_cast<uint32_t>(P.C));
    k.divH = FastDiv::make(static_cast<uint32_t>(P.H));
    k.divH2 = FastDiv::make(static_cast<uint32_t>(P.H2 > 0 ? P.H2 : 1));
    return k;
}

// A piece: tokens [t0, t0 + count) that are either whole batches (sp == S)
// or part of one batch (sp == count).
struct Piece {
    int64_t b0, s0, count, sp;
};

template <typename F>
rope_status_t for_each_piece(int64_t B, int64_t S, int64_t per_tok, F&& f) {
    const int64_t cap_tokens = int64_t(kMaxPieceTasks) / per_tok;  // >= 1
    if (B * S <= cap_tokens) return f(Piece{0, 0, B * S, S});
    if (S <= cap_tokens) {
        const int64_t nb = cap_tokens / S;
        for (int64_t b = 0; b < B; b += nb) {
            const int64_t cnt = (b + nb <= B ? nb : B - b) * S;
            rope_status_t st = f(Piece{b, 0, cnt, S});
            if (st != ROPE_OK) return st;
        }
        return ROPE_OK;
    }
    for (int64_t b = 0; b < B; ++b)
        for (int64_t s = 0; s < S; s += cap_tokens) {
            const int64_t cnt = s + cap_tokens <= S ? cap_tokens : S - s;
            rope_status_t st = f(Piece{b, s, cnt, cnt});
            if (st != ROPE_OK) return st;
        }
    return ROPE_OK;
}

int64_t grid_for(int64_t tasks, int64_t sms, int64_t blocks_per_sm, bool full) {
    const int64_t need = (tasks + kThreads - 1) / kThreads;
    const int64_t resident = sms * blocks_per_sm;
    return full || need < resident ? need : resident;
}

// Bytes spanned by a cos/sin tensor: the farthest row plus one row.
int64_t r_extent(const Resolved& R, int r, const int64_t* shape) {
    int64_t far = 0;
    for (int k = 0; k < 3; ++k) far += (shape[k] - 1) * R.rb[r][k];
    return far + R.L * R.e;
}

// Byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && pa < pb + uint64_t(nb) && pb < pa + uint64_t(na);
}

// x (or a gradient) is written in place while r1 and r2 are read: they must
// not share bytes (a tensor's bytes: x whole, cos/sin from their first to
// the end of their farthest row).
rope_status_t check_disjoint(const char* what, const void* x, int64_t xbytes, const void* r1,
                             const void* r2, const Resolved& R, const int64_t* r1_shape,
                             const int64_t* r2_shape) {
    if (overlaps(x, xbytes, r1, r_extent(R, 0, r1_shape)))
        return fail(ROPE_ERR_INVALID, "r1 (cos) overlaps %s, which is written in place", what);
    if (overlaps(x, xbytes, r2, r_extent(R, 1, r2_shape)))
        return fail(ROPE_ERR_INVALID, "r2 (sin) overlaps %s, which is written in place", what);
    return ROPE_OK;
}

// Plan, size and launch every piece of a validated call.
// The positions call's extra state: where the positions are and the
// frequency table.
struct PosCall {
    const int32_t* pos;
    int64_t pos_b, pos_s;  // element strides, 0 on broadcast dims
    FreqTable freq;
};

rope_status_t launch_all(int dir, int mode, int dtype, const Seg* seg, int nseg, const void* r1,
                         const void* r2, const Resolved& R, int64_t B, int64_t S,
                         rope_stream_t stream, const PosCall* pc_pos = nullptr,
                         bool host = false) {
    Plan P;
    rope_status_t st = make_plan(dir, mode, dtype, seg, nseg, r1, r2, R, &P, host, pc_pos != nullptr);
    if (st != ROPE_OK) return st;

    const char* err = nullptr;
    int sms = 0, bps = 0;
    if (device_sm_count(&sms, &err) != ROPE_OK) return fail(ROPE_ERR_CUDA, "%s", err);
    if (kernel_blocks_per_sm(P, &bps, &err) != ROPE_OK) return fail(ROPE_ERR_CUDA, "%s", err);
    if (bps < 1) bps = 1;

    KernelArgs whole = base_args(P, seg, nseg, r1, r2, R);
    if (pc_pos) {
        whole.pos = pc_pos->pos;
        whole.pos_b = pc_pos->pos_b;
        whole.pos_s = pc_pos->pos_s;
        whole.pairs = static_cast<int32_t>(R.L / 2);
    }
    const int64_t per_tok = int64_t(P.H + P.H2) * P.C;
    return for_each_piece(B, S, per_tok, [&](const Piece& pc) -> rope_status_t {
        KernelArgs k = whole;
        const int64_t t0 = pc.b0 * S + pc.s0;
        k.x += t0 * whole.tok_bytes;
        if (k.x2) k.x2 += t0 * whole.tok_bytes2;
        if (k.r1) k.r1 += pc.b0 * whole.r1_b + pc.s0 * whole.r1_s;
        if (k.r2) k.r2 += pc.b0 * whole.r2_b + pc.s0 * whole.r2_s;
        if (k.pos) k.pos += pc.b0 * whole.pos_b + pc.s0 * whole.pos_s;
        k.tasks = static_cast<uint32_t>(pc.count * per_tok);
        k.tasks1 = static_cast<uint32_t>(pc.count * int64_t(P.H) * P.C);
        k.divS = FastDiv::make(static_cast<uint32_t>(pc.sp));
        const uint32_t blocks = static_cast<uint32_t>(grid_for(k.tasks, sms, bps, P.full_grid));
        const char* e2 = nullptr;
        if (launch_piece(P, k, pc_pos ? &pc_pos->freq : nullptr, blocks, stream, &e2) != ROPE_OK)
            return fail(ROPE_ERR_CUDA, "%s", e2);
        return ROPE_OK;
    });
}

rope_status_t run(int dir, void* x, const void* r1, const void* r2, int dtype, int64_t B,
                  int64_t S, int64_t N, int64_t D, const int64_t* r1_shape,
                  const int64_t* r1_stride, const int64_t* r2_shape, const int64_t* r2_stride,
                  int64_t start, int64_t end, rope_stream_t stream, bool host_buffers,
                  int mode = kInterleave) {
    g_msg[0] = '\0';
    if (mode != kInterleave && mode != kHalf)
        return fail(ROPE_ERR_INVALID, "rotary mode %d is not interleave (1) or half (2)", mode);
    Resolved R;
    rope_status_t st = check(x, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                             r2_stride, start, end, &R);
    if (st != ROPE_OK || R.empty) return st;
    st = check_disjoint("x", x, B * S * N * D * R.e, r1, r2, R, r1_shape, r2_shape);
    if (st != ROPE_OK) return st;
    if (host_buffers) {
        // the kernel works on the host buffers in place: take the addresses
        // the device uses for them, or refuse a buffer it cannot reach
        const char* err = nullptr;
        const void* dx = nullptr;
        const void* d1 = nullptr;
        const void* d2 = nullptr;
        st = device_address(x, B * S * N * D * R.e, &dx, &err);
        if (st == ROPE_OK) st = device_address(r1, r_extent(R, 0, r1_shape), &d1, &err);
        if (st == ROPE_OK) st = device_address(r2, r_extent(R, 1, r2_shape), &d2, &err);
        if (st != ROPE_OK) return fail(st, "host buffer: %s", err);
        x = const_cast<void*>(dx);
        r1 = d1;
        r2 = d2;
    }
    const Seg seg{x, N, D, start};
    return launch_all(dir, mode, dtype, &seg, 1, r1, r2, R, B, S, stream, nullptr, host_buffers);
}

// The fused query + key call: both tensors share B, S and each token's
// cos/sin row (r1/r2 of shape (Br, Sr, 1, L)); the slices have one length L.
rope_status_t run_qk(int dir, void* q, void* k, const void* r1, const void* r2, int dtype,
                     int64_t B, int64_t S, int64_t Nq, int64_t Dq, int64_t q_start, int64_t q_end,
                     int64_t Nk, int64_t Dk, int64_t k_start, int64_t k_end,
                     const int64_t* r1_shape, const int64_t* r1_stride, const int64_t* r2_shape,
                     const int64_t* r2_stride, rope_stream_t stream) {
    g_msg[0] = '\0';
    if ((q_end - q_start) != (k_end - k_start))
        return fail(ROPE_ERR_INVALID, "query slice length %lld and key slice length %lld differ",
                    (long long)(q_end - q_start), (long long)(k_end - k_start));
    if ((r1_shape && r1_shape[2] != 1) || (r2_shape && r2_shape[2] != 1))
        return fail(ROPE_ERR_INVALID, "the fused query + key call shares one cos/sin row per "
                    "token: r1 and r2 must have size 1 in the head dim");
    Resolved Rq, Rk;
    rope_status_t st = check(q, r1, r2, dtype, B, S, Nq, Dq, r1_shape, r1_stride, r2_shape,
                             r2_stride, q_start, q_end, &Rq);
    if (st != ROPE_OK) return fail_prefixed(st, "query");
    st = check(k, r1, r2, dtype, B, S, Nk, Dk, r1_shape, r1_stride, r2_shape, r2_stride, k_start,
               k_end, &Rk);
    if (st != ROPE_OK) return fail_prefixed(st, "key");
    // q and k are both written: they must not share a byte, nor may either
    // share one with r1 / r2
    const int64_t qbytes = Rq.empty ? 0 : B * S * Nq * Dq * Rq.e;
    const int64_t kbytes = Rk.empty ? 0 : B * S * Nk * Dk * Rk.e;
    if (overlaps(q, qbytes, k, kbytes))
        return fail(ROPE_ERR_INVALID, "query and key overlap; both are written in place");
    if (!Rq.empty && (st = check_disjoint("the query", q, qbytes, r1, r2, Rq, r1_shape, r2_shape)) != ROPE_OK)
        return st;
    if (!Rk.empty && (st = check_disjoint("the key", k, kbytes, r1, r2, Rk, r1_shape, r2_shape)) != ROPE_OK)
        return st;
    Seg seg[2];
    int nseg = 0;
    if (!Rq.empty) seg[nseg++] = Seg{q, Nq, Dq, q_start};
    if (!Rk.empty) seg[nseg++] = Seg{k, Nk, Dk, k_start};
    if (nseg == 0) return ROPE_OK;
    return launch_all(dir, kInterleave, dtype, seg, nseg, r1, r2, Rq.empty ? Rk : Rq, B, S, stream);
}

// The positions call: cos/sin of theta_k = p * base^(-2k/L) computed in
// the kernel from one int32 position per (b, s).
rope_status_t run_pos(int dir, void* x, const int32_t* positions, int dtype, int64_t B, int64_t S,
                      int64_t N, int64_t D, const int64_t* pos_shape, const int64_t* pos_stride,
                      double base, int64_t start, int64_t end, int mode, rope_stream_t stream) {
    g_msg[0] = '\0';
    if (mode != kInterleave && mode != kHalf)
        return fail(ROPE_ERR_INVALID, "rotary mode %d is not interleave (1) or half (2)", mode);
    if (!(base > 0.0) || !isfinite(base))
        return fail(ROPE_ERR_INVALID, "base %g must be a finite number > 0", base);
    // the x rules are those of the table call; a stand-in table of shape
    // (1, 1, 1, L) lets check() apply them
    const int64_t L = end - start;
    const int64_t ones[4] = {1, 1, 1, L >= 0 ? L : 0};
    const int64_t unit[4] = {0, 0, 0, 1};
    Resolved R;
    rope_status_t st = check(x, x, x, dtype, B, S, N, D, ones, unit, ones, unit, start, end, &R);
    if (st != ROPE_OK || R.empty) return st;
    if (!positions) return fail(ROPE_ERR_NULLPTR, "positions is null");
    if (!pos_shape || !pos_stride) return fail(ROPE_ERR_NULLPTR, "pos_shape or pos_stride is null");
    const int64_t xdim[2] = {B, S};
    int64_t ps[2];
    for (int k = 0; k < 2; ++k) {
        if (!(pos_shape[k] == 1 || pos_shape[k] == xdim[k]))
            return fail(ROPE_ERR_INVALID, "positions dim %d is %lld; it must be 1 or %lld", k,
                        (long long)pos_shape[k], (long long)xdim[k]);
        if (pos_shape[k] != 1 && pos_stride[k] < 0)
            return fail(ROPE_ERR_INVALID, "positions stride %d is negative", k);
        ps[k] = pos_shape[k] == 1 ? 0 : pos_stride[k];
    }
    if (reinterpret_cast<uintptr_t>(positions) % 4)
        return fail(ROPE_ERR_INVALID, "positions must be 4-byte aligned int32");
    if (L / 2 > kMaxPairs)
        return fail(ROPE_ERR_INVALID, "slice length %lld exceeds %d", (long long)L, 2 * kMaxPairs);

    PosCall pc{};
    pc.pos = positions;
    pc.pos_b = ps[0];
    pc.pos_s = ps[1];
    for (int64_t k = 0; k < L / 2; ++k) {
        const double w = pow(base, -2.0 * double(k) / double(L));
        pc.freq.hi[k] = static_cast<float>(w);
        pc.freq.lo[k] = static_cast<float>(w - static_cast<double>(pc.freq.hi[k]));
    }
    const Seg seg{x, N, D, start};
    return launch_all(dir, mode, dtype, &seg, 1, nullptr, nullptr, R, B, S, stream, &pc);
}

}  // namespace
}  // namespace rope

extern "C" {

rope_status_t rope_partial_inplace_fwd(void* x, const void* r1, const void* r2,
                                       rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                       int64_t D, const int64_t r1_shape[4],
                                       const int64_t r1_stride[4], const int64_t r2_shape[4],
                                       const int64_t r2_stride[4], int64_t start, int64_t end,
                                       rope_stream_t stream) {
    return rope::run(rope::kFwd, x, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                     r2_stride, start, end, stream, false);
}

rope_status_t rope_partial_inplace_bwd(void* grad, const void* r1, const void* r2,
                                       rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                       int64_t D, const int64_t r1_shape[4],
                                       const int64_t r1_stride[4], const int64_t r2_shape[4],
                                       const int64_t r2_stride[4], int64_t start, int64_t end,
                                       rope_stream_t stream) {
    return rope::run(rope::kBwd, grad, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                     r2_stride, start, end, stream, false);
}

rope_status_t rope_partial_inplace_fwd_mode(void* x, const void* r1, const void* r2,
                                            rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                            int64_t D, const int64_t r1_shape[4],
                                            const int64_t r1_stride[4], const int64_t r2_shape[4],
                                            const int64_t r2_stride[4], int64_t start,
                                            int64_t end, rope_mode_t mode, rope_stream_t stream) {
    return rope::run(rope::kFwd, x, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                     r2_stride, start, end, stream, false, mode);
}

rope_status_t rope_partial_inplace_bwd_mode(void* grad, const void* r1, const void* r2,
                                            rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                            int64_t D, const int64_t r1_shape[4],
                                            const int64_t r1_stride[4], const int64_t r2_shape[4],
                                            const int64_t r2_stride[4], int64_t start,
                                            int64_t end, rope_mode_t mode, rope_stream_t stream) {
    return rope::run(rope::kBwd, grad, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                     r2_stride, start, end, stream, false, mode);
}

rope_status_t rope_partial_inplace_fwd_pos(void* x, const int32_t* positions, rope_dtype_t dtype,
                                           int64_t B, int64_t S, int64_t N, int64_t D,
                                           const int64_t pos_shape[2], const int64_t pos_stride[2],
                                           double base, int64_t start, int64_t end,
                                           rope_mode_t mode, rope_stream_t stream) {
    return rope::run_pos(rope::kFwd, x, positions, dtype, B, S, N, D, pos_shape, pos_stride, base,
                         start, end, mode, stream);
}

rope_status_t rope_partial_inplace_bwd_pos(void* grad, const int32_t* positions,
                                           rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                           int64_t D, const int64_t pos_shape[2],
                                           const int64_t pos_stride[2], double base,
                                           int64_t start, int64_t end, rope_mode_t mode,
                                           rope_stream_t stream) {
    return rope::run_pos(rope::kBwd, grad, positions, dtype, B, S, N, D, pos_shape, pos_stride,
                         base, start, end, mode, stream);
}

rope_status_t rope_partial_inplace_fwd_qk(void* q, void* k, const void* r1, const void* r2,
                                          rope_dtype_t dtype, int64_t B, int64_t S, int64_t Nq,
                                          int64_t Dq, int64_t q_start, int64_t q_end, int64_t Nk,
                                          int64_t Dk, int64_t k_start, int64_t k_end,
                                          const int64_t r1_shape[4], const int64_t r1_stride[4],
                                          const int64_t r2_shape[4], const int64_t r2_stride[4],
                                          rope_stream_t stream) {
    return rope::run_qk(rope::kFwd, q, k, r1, r2, dtype, B, S, Nq, Dq, q_start, q_end, Nk, Dk,
                        k_start, k_end, r1_shape, r1_stride, r2_shape, r2_stride, stream);
}

rope_status_t rope_partial_inplace_bwd_qk(void* dq, void* dk, const void* r1, const void* r2,
                                          rope_dtype_t dtype, int64_t B, int64_t S, int64_t Nq,
                                          int64_t Dq, int64_t q_start, int64_t q_end, int64_t Nk,
                                          int64_t Dk, int64_t k_start, int64_t k_end,
                                          const int64_t r1_shape[4], const int64_t r1_stride[4],
                                          const int64_t r2_shape[4], const int64_t r2_stride[4],
                                          rope_stream_t stream) {
    return rope::run_qk(rope::kBwd, dq, dk, r1, r2, dtype, B, S, Nq, Dq, q_start, q_end, Nk, Dk,
                        k_start, k_end, r1_shape, r1_stride, r2_shape, r2_stride, stream);
}

rope_status_t rope_partial_inplace_fwd_host(void* x, const void* r1, const void* r2,
                                            rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                            int64_t D, const int64_t r1_shape[4],
                                            const int64_t r1_stride[4], const int64_t r2_shape[4],
                                            const int64_t r2_stride[4], int64_t start,
                                            int64_t end, rope_stream_t stream) {
    return rope::run(rope::kFwd, x, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                     r2_stride, start, end, stream, true);
}

rope_status_t rope_partial_inplace_bwd_host(void* grad, const void* r1, const void* r2,
                                            rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                            int64_t D, const int64_t r1_shape[4],
                                            const int64_t r1_stride[4], const int64_t r2_shape[4],
                                            const int64_t r2_stride[4], int64_t start,
                                            int64_t end, rope_stream_t stream) {
    return rope::run(rope::kBwd, grad, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                     r2_stride, start, end, stream, true);
}

rope_status_t rope_partial_token_shard(int64_t B, int64_t S, int32_t rank, int32_t world,
                                       int64_t* t0, int64_t* t1, rope_token_run_t runs[3],
                                       int32_t* nruns) {
    using namespace rope;
    g_msg[0] = '\0';
    if (!t0 || !t1 || !runs || !nruns) return fail(ROPE_ERR_NULLPTR, "an output pointer is null");
    if (B < 0 || S < 0)
        return fail(ROPE_ERR_INVALID, "negative size: B=%lld S=%lld", (long long)B, (long long)S);
    if (world < 1 || rank < 0 || rank >= world)
        return fail(ROPE_ERR_INVALID, "rank %d is outside [0, world=%d)", (int)rank, (int)world);
    if (mul_overflows(B, S))
        return fail(ROPE_ERR_INVALID, "B=%lld x S=%lld tokens overflow", (long long)B, (long long)S);
    const int64_t T = B * S;
    // balanced: the first T % world ranks take one token more
    const int64_t base = T / world, rem = T % world;
    const int64_t lo = int64_t(rank) * base + (rank < rem ? rank : rem);
    const int64_t hi = lo + base + (rank < rem ? 1 : 0);
    *t0 = lo;
    *t1 = hi;
    *nruns = 0;
    if (lo == hi) return ROPE_OK;
    int64_t t = lo;
    if (t % S != 0) {  // the rest of the batch the range enters mid-way
        const int64_t s = t % S, n = (S - s < hi - t) ? S - s : hi - t;
        runs[(*nruns)++] = rope_token_run_t{t / S, s, 1, n};
        t += n;
    }
    if (hi - t >= S) {  // whole batches
        const int64_t nb = (hi - t) / S;
        runs[(*nruns)++] = rope_token_run_t{t / S, 0, nb, S};
        t += nb * S;
    }
    if (t < hi) {  // the start of the batch the range leaves mid-way
        runs[(*nruns)++] = rope_token_run_t{t / S, 0, 1, hi - t};
        t = hi;
    }
    return ROPE_OK;
}

const char* rope_status_str(rope_status_t status) {
    switch (status) {
        case ROPE_OK: return "ROPE_OK";
        case ROPE_ERR_NULLPTR: return "ROPE_ERR_NULLPTR";
        case ROPE_ERR_INVALID: return "ROPE_ERR_INVALID";
        case ROPE_ERR_CUDA: return "ROPE_ERR_CUDA";
    }
    return "ROPE_ERR_UNKNOWN";
}

const char* rope_last_error_message(void) { return rope::g_msg; }

rope_status_t rope_partial_plan_mode(const void* x, const void* r1, const void* r2,
                                     rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                     int64_t D, const int64_t r1_shape[4],
                                     const int64_t r1_stride[4], const int64_t r2_shape[4],
                                     const int64_t r2_stride[4], int64_t start, int64_t end,
                                     rope_mode_t mode, int32_t sm_count, rope_plan_t* plan) {
    using namespace rope;
    g_msg[0] = '\0';
    if (!plan) return fail(ROPE_ERR_NULLPTR, "plan is null");
    *plan = rope_plan_t{};
    const int m = static_cast<int>(mode);
    if (m != kInterleave && m != kHalf)
        return fail(ROPE_ERR_INVALID, "rotary mode %d is not interleave (1) or half (2)", m);
    Resolved R;
    rope_status_t st = check(x, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                             r2_stride, start, end, &R);
    if (st != ROPE_OK || R.empty) return st;
    Plan P;
    const Seg seg{const_cast<void*>(x), N, D, start};
    st = make_plan(kFwd, m, dtype, &seg, 1, r1, r2, R, &P);
    if (st != ROPE_OK) return st;
    if (!kernel_lookup(P))
        return fail(ROPE_ERR_CUDA, "internal error: no kernel instance for this plan");
    int sms = sm_count, bps = kBlocksPerSmCap;
    if (sm_count <= 0) {
        const char* err = nullptr;
        if (device_sm_count(&sms, &err) != ROPE_OK) return fail(ROPE_ERR_CUDA, "%s", err);
        if (kernel_blocks_per_sm(P, &bps, &err) != ROPE_OK) return fail(ROPE_ERR_CUDA, "%s", err);
    }
    const int64_t per_tok = int64_t(P.H + P.H2) * P.C;
    int64_t max_blocks = 0, launches = 0;
    for_each_piece(B, S, per_tok, [&](const Piece& pc) -> rope_status_t {
        const int64_t g = grid_for(pc.count * per_tok, sms, bps, P.full_grid);
        if (g > max_blocks) max_blocks = g;
        ++launches;
        return ROPE_OK;
    });
    plan->path = P.lanes ? 3 : P.path;  // kOddPair reports 4
    plan->vec_bytes = P.vec;
    plan->heads_per_thread = P.U;
    plan->threads_per_block = kThreads;
    plan->blocks = max_blocks;
    plan->tasks = B * S * per_tok;
    plan->chunks_per_row = P.C;
    plan->r_per_head = P.r_head ? 1 : 0;
    plan->launches = launches;
    return ROPE_OK;
}

rope_status_t rope_partial_plan(const void* x, const void* r1, const void* r2,
                                rope_dtype_t dtype, int64_t B, int64_t S, int64_t N, int64_t D,
                                const int64_t r1_shape[4], const int64_t r1_stride[4],
                                const int64_t r2_shape[4], const int64_t r2_stride[4],
                                int64_t start, int64_t end, int32_t sm_count,
                                rope_plan_t* plan) {
    return rope_partial_plan_mode(x, r1, r2, dtype, B, S, N, D, r1_shape, r1_stride, r2_shape,
                                  r2_stride, start, end, ROPE_MODE_INTERLEAVE, sm_count, plan);
}

}  // extern "C"

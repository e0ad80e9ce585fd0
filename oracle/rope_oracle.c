/*
 * rope_oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, scalar CPU statement of the in-place partial interleaved
 * rotary position embedding (inplace_partial_rotary_mul) and its backward.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  It shares no code, header, table or constant
 * with the CUDA path.
 *
 * Sources (the pages this follows):
 *   [P1] "CANN ops-transformer inplace_partial_rotary_mul" (mhpn.cn/news/2302710)
 *        section "功能与计算公式" (formula: x1 = x_slice[..., ::2],
 *        x2 = x_slice[..., 1::2], x_rotate = cat(-x2, x1),
 *        x_out = x_slice*cos + x_rotate*sin, written back to x[..., start:end]);
 *        same section, kernel evidence (Process: ComputeMul x*cos, Gather with
 *        index i^1, ComputeMul *sin, InterleavedInversion with mask
 *        0x5555555555555555, Add);
 *        section "Tiling 与 Kernel 的工程细节" (non-fp32 inputs are cast to
 *        FP32 for the multiply-adds and written back with CAST_RINT).
 *   [P3] "ANE实战 RoPE位置编码在MIL中的纯ANE实现" (lpnh.cn/news/2229363)
 *        section "反向传播" (the backward is the inverse rotation of the
 *        gradient, applied in place).
 *
 * Precision: [P1] fixes it -- every product and the sum are single IEEE
 * binary32 operations (round to nearest even), computed as separate
 * statements.  This file must be compiled with -ffp-contract=off so the
 * compiler cannot fuse a multiply and an add.
 *
 * Readings taken where the pages are silent or garbled:
 *   - "cat(-x2, x1)" in interleave mode is an interleave: the rotated vector
 *     holds -x[2i+1] in lane 2i and x[2i] in lane 2i+1 (the i^1 gather).
 *   - The inversion mask 0x5555... sets bits 0,2,4,...: it negates the
 *     0-based EVEN lanes of the swapped product.
 *   - Pairs are counted from `start` (slice-relative), so any start is legal
 *     as long as end-start is even.
 *   - The backward is the exact transpose of the forward's per-lane Jacobian:
 *     dx[2i]   = g[2i]c[2i]     + g[2i+1]s[2i+1]
 *     dx[2i+1] = g[2i+1]c[2i+1] - g[2i]s[2i]
 *     with the products rounded first, then one rounded add.  With a
 *     pair-duplicated table this is [P3]'s inverse rotation.
 *   - Half-split mode (a second rotary mode): x1 and x2 are the first and
 *     second halves of the slice and x_rotate = cat(-x2, x1) read literally,
 *     which is [P3]'s rotate_half ("swap the two halves, negate the front
 *     half"): lane j pairs with lane j + L/2, and the formulas above hold
 *     with (2i, 2i+1) replaced by (j, j + L/2).
 *
 * Storage conversions (binary16 and bfloat16 to and from binary32) are
 * written out from the IEEE 754 definitions of the formats below; they call
 * no library conversion.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* storage type codes, the same numbering the tests pass in */
enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_FP32 = 2 };
/* formulation codes */
enum { ORC_GATHER_CHAIN = 0, ORC_PAIR_ROTATION = 1 };
/* direction codes */
enum { ORC_FWD = 0, ORC_BWD = 1 };
/* rotary modes (the interleave code is the ACLNN value 1) */
enum { ORC_INTERLEAVE = 1, ORC_HALF = 2 };

/* ------------------------------------------------------------------------ */
/* Format conversions from the IEEE 754 definitions.                        */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/*
 * Round a binary32 value to a narrower binary format with `mant` explicit
 * fraction bits, minimum normal exponent `emin`, maximum exponent `emax`
 * and exponent bias `bias`, round-to-nearest-ties-to-even, gradual
 * underflow, overflow to infinity.  Returns the format's bit pattern.
 *
 * Method: write |v| = m * 2^E exactly (m an integer of at most 24 bits).
 * The target's spacing at v is 2^Q with Q = max(floor(log2|v|), emin) - mant.
 * Divide m*2^E by 2^Q, rounding the quotient n to the nearest integer (ties
 * to even).  Then v rounds to n * 2^Q; encode n.
 */
static uint32_t round_from_f32(float v, int mant, int emin, int emax, int bias,
                               int total_bits)
{
    const uint32_t u = f32_bits(v);
    const uint32_t sign = (u >> 31) & 1u;
    const uint32_t efield = (u >> 23) & 0xffu;
    const uint32_t frac = u & 0x7fffffu;
    const uint32_t exp_all_ones = (1u << (total_bits - 1 - mant)) - 1u;
    const uint32_t sign_out = sign << (total_bits - 1);

    if (efield == 0xffu) {
        if (frac != 0) /* NaN stays NaN: quiet bit plus any top payload bits */
            return sign_out | (exp_all_ones << mant) | (1u << (mant - 1)) |
                   (frac >> (23 - mant));
        return sign_out | (exp_all_ones << mant); /* infinity */
    }
    if (efield == 0 && frac == 0)
        return sign_out; /* signed zero */

    /* exact integer significand and exponent of |v| */
    uint64_t m;
    int E;
    int e_unb; /* floor(log2 |v|) */
    if (efield == 0) {
        /* subnormal: |v| = frac * 2^-149; with nbits the bit length of frac,
           floor(log2|v|) = (nbits - 1) - 149 */
        int nbits = 0;
        for (uint32_t t = frac; t; t >>= 1) nbits++;
        m = frac;
        E = -149;
        e_unb = nbits - 150;
    } else {
        m = (uint64_t)frac | 0x800000u;
        E = (int)efield - 150;
        e_unb = (int)efield - 127;
    }

    if (e_unb > emax)
        return sign_out | (exp_all_ones << mant); /* beyond the format: inf */

    const int Q = (e_unb > emin ? e_unb : emin) - mant;
    const int shift = Q - E;
    uint64_t n;
    if (shift <= 0) {
        n = m << (-shift); /* exact: v is a multiple of the spacing */
    } else if (shift >= 40) {
        n = 0; /* far below half the smallest spacing */
    } else {
        const uint64_t rem = m & ((1ull << shift) - 1ull);
        const uint64_t half = 1ull << (shift - 1);
        n = m >> shift;
        if (rem > half || (rem == half && (n & 1ull)))
            n += 1;
    }

    /* encode n * 2^Q */
    uint32_t out;
    if (Q == emin - mant) {
        /* subnormal spacing: n < 2^mant is a subnormal; n == 2^mant is the
           smallest normal, whose encoding is the same integer. Larger n only
           happen when e_unb == emin, handled by the normal branch below. */
        if (n <= (1ull << mant)) {
            out = (uint32_t)n;
            return sign_out | out;
        }
    }
    /* normal: n in [2^mant, 2^(mant+1)]; n == 2^(mant+1) carries into the
       exponent through the addition */
    const int e_q = Q + mant; /* unbiased exponent of the binade */
    out = ((uint32_t)(e_q + bias) << mant) + (uint32_t)(n - (1ull << mant));
    if ((out >> mant) >= exp_all_ones)
        out = exp_all_ones << mant; /* rounded up past the largest finite */
    return sign_out | out;
}

uint16_t oracle_f32_to_bf16(float v) { return (uint16_t)round_from_f32(v, 7, -126, 127, 127, 16); }
uint16_t oracle_f32_to_f16(float v) { return (uint16_t)round_from_f32(v, 10, -14, 15, 15, 16); }

/* bfloat16 is the top half of a binary32 pattern: widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* binary16 -> binary32 from the format definition. */
float oracle_f16_to_f32(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int efield = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    float mag;
    if (efield == 0x1f) {
        if (frac) {
            /* NaN: carry the payload into the binary32 fraction */
            return bits_f32(((uint32_t)sign << 31) | 0x7fc00000u | ((uint32_t)frac << 13));
        }
        mag = INFINITY;
    } else if (efield == 0) {
        mag = ldexpf((float)frac, -24); /* subnormal: frac * 2^-24 */
    } else {
        mag = ldexpf((float)(frac | 0x400), efield - 25); /* (1024+frac) * 2^(e-15-10) */
    }
    return sign ? -mag : mag;
}

/* Batch versions for the tests. */
void oracle_f32_to_bf16_n(const float* in, uint16_t* out, int64_t n)
{ for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_bf16(in[i]); }
void oracle_f32_to_f16_n(const float* in, uint16_t* out, int64_t n)
{ for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_f16(in[i]); }
void oracle_bf16_to_f32_n(const uint16_t* in, float* out, int64_t n)
{ for (int64_t i = 0; i < n; i++) out[i] = oracle_bf16_to_f32(in[i]); }
void oracle_f16_to_f32_n(const uint16_t* in, float* out, int64_t n)
{ for (int64_t i = 0; i < n; i++) out[i] = oracle_f16_to_f32(in[i]); }

/* ------------------------------------------------------------------------ */
/* Element access in the storage type.                                      */
/* ------------------------------------------------------------------------ */

static float load_elem(const void* base, int64_t idx, int dtype)
{
    if (dtype == ORC_FP32) return ((const float*)base)[idx];
    const uint16_t h = ((const uint16_t*)base)[idx];
    return dtype == ORC_BF16 ? oracle_bf16_to_f32(h) : oracle_f16_to_f32(h);
}

/* CAST_RINT: one rounding from binary32 to the storage type. */
static void store_elem(void* base, int64_t idx, float v, int dtype)
{
    if (dtype == ORC_FP32) { ((float*)base)[idx] = v; return; }
    ((uint16_t*)base)[idx] = dtype == ORC_BF16 ? oracle_f32_to_bf16(v) : oracle_f32_to_f16(v);
}

/* ------------------------------------------------------------------------ */
/* One slice row.                                                           */
/* ------------------------------------------------------------------------ */

/*
 * [P1] kernel op chain, forward, on one slice of L lanes:
 *   t1[j] = x[j] * c[j]                   (ComputeMul with cos)
 *   g[j]  = x[j ^ 1]                      (Gather, index table j^1)
 *   t2[j] = g[j] * s[j]                   (ComputeMul with sin)
 *   t2[j] = -t2[j]   for even j           (InterleavedInversion, mask 0x5555...)
 *   y[j]  = t1[j] + t2[j]                 (Add)
 * Backward, the transposed chain on the gradient:
 *   t1[j] = g[j] * c[j];  w[j] = u[j ^ 1] with u[k] = g[k] * s[k];
 *   w[j] = -w[j] for odd j;  dx[j] = t1[j] + w[j]
 * Half-split mode: the gather index is j + L/2 (first half) or j - L/2
 * (second half); the forward negates the first half of the swapped
 * product, the backward the second half.
 */
static int64_t partner(int mode, int64_t j, int64_t L)
{
    if (mode == ORC_INTERLEAVE) return j ^ 1;
    return j < L / 2 ? j + L / 2 : j - L / 2;
}

static int negated(int mode, int dir, int64_t j, int64_t L)
{
    const int first = mode == ORC_INTERLEAVE ? (j % 2 == 0) : (j < L / 2);
    return dir == ORC_FWD ? first : !first;
}

static void row_gather_chain(int dir, int mode, float* v, const float* c, const float* s,
                             float* t1, float* t2, int64_t L)
{
    int64_t j;
    if (dir == ORC_FWD) {
        for (j = 0; j < L; j++) t1[j] = v[j] * c[j];
        for (j = 0; j < L; j++) t2[j] = v[partner(mode, j, L)] * s[j];
        for (j = 0; j < L; j++) if (negated(mode, dir, j, L)) t2[j] = -t2[j];
    } else {
        for (j = 0; j < L; j++) t1[j] = v[j] * c[j];
        for (j = 0; j < L; j++) t2[j] = v[partner(mode, j, L)] * s[partner(mode, j, L)];
        for (j = 0; j < L; j++) if (negated(mode, dir, j, L)) t2[j] = -t2[j];
    }
    for (j = 0; j < L; j++) v[j] = t1[j] + t2[j];
}

/*
 * The same result written as one 2x2 rotation per pair (the explicit pair form),
 * lanes (m, n) = (2i, 2i+1) in interleave mode, (i, i + L/2) in half mode:
 *   fwd: y_m = x_m c_m - x_n s_m ;  y_n = x_n c_n + x_m s_n
 *   bwd: d_m = g_m c_m + g_n s_n ;  d_n = g_n c_n - g_m s_m
 */
static void row_pair_rotation(int dir, int mode, float* v, const float* c, const float* s,
                              int64_t L)
{
    for (int64_t k = 0; k < L / 2; k++) {
        const int64_t i = mode == ORC_INTERLEAVE ? 2 * k : k;
        const int64_t n = mode == ORC_INTERLEAVE ? 2 * k + 1 : k + L / 2;
        const float a = v[i], b = v[n];
        float p, q, r, t;
        if (dir == ORC_FWD) {
            p = a * c[i];  q = b * s[i];  v[i] = p - q;
            r = b * c[n]; t = a * s[n]; v[n] = r + t;
        } else {
            p = a * c[i];  q = b * s[n];  v[i] = p + q;
            r = b * c[n]; t = a * s[i];   v[n] = r - t;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* The whole tensor.                                                        */
/* ------------------------------------------------------------------------ */

/*
 * oracle_rope: apply the forward (dir 0) or backward (dir 1) in place to
 * the contiguous BSND tensor x (storage type `dtype`), rotating only lanes
 * [start, end) of each row, pairing lanes in `mode` (1 interleave, 2 half).  r1 holds cos, r2 holds sin, each of shape
 * (rX_shape[0..3]) with element strides rX_stride[0..3]; a dimension of size
 * 1 broadcasts.  formulation selects the gather chain (0) or the pair
 * rotation (1).  Returns 0, or -1 on arguments it does not accept (the
 * oracle checks only what it needs to stay in bounds).
 */
int oracle_rope_mixed(int dir, int formulation, int mode, int dtype, int r_dtype, void* x,
                      const void* r1, const void* r2, int64_t B, int64_t S, int64_t N, int64_t D,
                      const int64_t* r1_shape, const int64_t* r1_stride,
                      const int64_t* r2_shape, const int64_t* r2_stride,
                      int64_t start, int64_t end);

int oracle_rope(int dir, int formulation, int mode, int dtype, void* x, const void* r1,
                const void* r2, int64_t B, int64_t S, int64_t N, int64_t D,
                const int64_t* r1_shape, const int64_t* r1_stride,
                const int64_t* r2_shape, const int64_t* r2_stride,
                int64_t start, int64_t end)
{
    return oracle_rope_mixed(dir, formulation, mode, dtype, dtype, x, r1, r2, B, S, N, D,
                             r1_shape, r1_stride, r2_shape, r2_stride, start, end);
}

/*
 * oracle_rope_mixed: as oracle_rope, with cos/sin stored in their own type
 * r_dtype (the in-kernel cos/sin of the positions call are fp32 values while
 * x may be bf16 or fp16).
 */
int oracle_rope_mixed(int dir, int formulation, int mode, int dtype, int r_dtype, void* x,
                      const void* r1, const void* r2, int64_t B, int64_t S, int64_t N, int64_t D,
                      const int64_t* r1_shape, const int64_t* r1_stride,
                      const int64_t* r2_shape, const int64_t* r2_stride,
                      int64_t start, int64_t end)
{
    const int64_t L = end - start;
    if (B < 0 || S < 0 || N < 0 || D < 0 || start < 0 || end > D || L < 0 || (L & 1))
        return -1;
    if (mode != ORC_INTERLEAVE && mode != ORC_HALF)
        return -1;
    if (L == 0 || B == 0 || S == 0 || N == 0)
        return 0; /* [P1]: an empty slice or empty tensor leaves x unchanged */
    const int64_t xdim[3] = {B, S, N};
    for (int k = 0; k < 3; k++) {
        if (!(r1_shape[k] == 1 || r1_shape[k] == xdim[k])) return -1;
        if (!(r2_shape[k] == 1 || r2_shape[k] == xdim[k])) return -1;
    }
    if (r1_shape[3] != L || r2_shape[3] != L) return -1;

    float* v = (float*)malloc(sizeof(float) * (size_t)L);
    float* c = (float*)malloc(sizeof(float) * (size_t)L);
    float* s = (float*)malloc(sizeof(float) * (size_t)L);
    float* t1 = (float*)malloc(sizeof(float) * (size_t)L);
    float* t2 = (float*)malloc(sizeof(float) * (size_t)L);
    if (!v || !c || !s || !t1 || !t2) { free(v); free(c); free(s); free(t1); free(t2); return -1; }

    for (int64_t b = 0; b < B; b++)
        for (int64_t si = 0; si < S; si++)
            for (int64_t n = 0; n < N; n++) {
                const int64_t row = ((b * S + si) * N + n) * D + start;
                /* a broadcast dimension (size 1) always indexes 0 */
                const int64_t o1 = (r1_shape[0] == 1 ? 0 : b) * r1_stride[0] +
                                   (r1_shape[1] == 1 ? 0 : si) * r1_stride[1] +
                                   (r1_shape[2] == 1 ? 0 : n) * r1_stride[2];
                const int64_t o2 = (r2_shape[0] == 1 ? 0 : b) * r2_stride[0] +
                                   (r2_shape[1] == 1 ? 0 : si) * r2_stride[1] +
                                   (r2_shape[2] == 1 ? 0 : n) * r2_stride[2];
                for (int64_t j = 0; j < L; j++) {
                    v[j] = load_elem(x, row + j, dtype);
                    c[j] = load_elem(r1, o1 + j * r1_stride[3], r_dtype);
                    s[j] = load_elem(r2, o2 + j * r2_stride[3], r_dtype);
                }
                if (formulation == ORC_GATHER_CHAIN)
                    row_gather_chain(dir, mode, v, c, s, t1, t2, L);
                else
                    row_pair_rotation(dir, mode, v, c, s, L);
                for (int64_t j = 0; j < L; j++) store_elem(x, row + j, v[j], dtype);
            }
    free(v); free(c); free(s); free(t1); free(t2);
    return 0;
}

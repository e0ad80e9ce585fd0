// rope_kernels.cuh -- the sm_103a kernels of the in-place partial rotary
// embedding, forward and backward, for bf16 / fp16 / fp32 storage:
//   rope_partial_kernel      one tensor, interleaved pairs (the page's mode)
//   rope_partial_half_kernel one tensor, half-split pairs (i, i + L/2)
//   rope_partial_half_lanes_kernel  the same when a row's accesses fit one
//                            warp: the partner access comes by warp shuffle
//   rope_partial_qk_kernel   query and key in one launch, one cos/sin row
//   rope_partial_pos_kernel  cos/sin computed from positions (no table)
//   rope_partial_odd_kernel  16-bit interleave with an odd start: a lane
//                            per aligned word, straddling halves by shuffle
//
// What it computes ("CANN ops-transformer inplace_partial_rotary_mul",
// section 功能与计算公式, and its kernel op chain): for every row
// (b, s, n) of a BSND tensor and every pair (2i, 2i+1) of the slice
// [start, end) counted from start,
//   forward : y0 = x0*c0 - x1*s0          y1 = x1*c1 + x0*s1
//   backward: d0 = g0*c0 + g1*s1          d1 = g1*c1 - g0*s0
// Inputs are widened to fp32, each product and each sum is one fp32 rounding
// (__fmul_rn / __fadd_rn / __fsub_rn, which the compiler never contracts
// into an FMA), and the result is rounded once to the storage type with
// round-to-nearest-even (the page's CAST_RINT write-back).
//
// How (GB300): the op is a streaming read-modify-write of the slice bytes,
// bound by HBM bandwidth, so there is no tensor-core work and no shared
// memory (except the positions kernel's 4 KB frequency table).  One work
// item is (token, head group, chunk):
//   * a chunk is one 16-, 8- or 4-byte access of x that holds whole pairs,
//     so the pair swap happens inside a thread's registers (no shuffles);
//     rows whose slice is not aligned for that fall back to a scalar path
//     with one access per element ("scalar pair"); in half-split mode a
//     chunk's partner lies L/2 lanes on: in another lane of the warp when
//     the row's chunks fit one warp (a shuffle brings it), otherwise in the
//     same thread; a 16-bit slice with an odd start has its pairs straddle
//     aligned words, and rows of up to 32 pairs then take a lane per word
//     with the straddling halves brought by shuffle;
//   * a thread keeps the chunk's cos/sin in registers and walks U
//     consecutive heads of the same token (heads hg*U .. hg*U + U - 1),
//     issuing all U loads of x before any arithmetic, so U accesses per
//     thread are in flight and the cos/sin bytes are read once per U heads;
//   * consecutive threads take consecutive chunks of a row, so a warp reads
//     whole 32-byte sectors of each row's slice;
//   * the flat work index is split by three multiply-high divisions per
//     item; the grid usually covers it once (one block per 256 items, so
//     the hardware starts a block as each one ends), and for the cases that
//     measured faster that way it is sized to the resident blocks of all
//     SMs and strides over the work (the host picks per access kind);
//   * launches use programmatic dependent launch: every kernel waits on
//     griddepcontrol before its first global access, so only its launch and
//     ramp overlap the tail of the kernel before it in the stream.
// Only slice bytes are read or written; every other byte of x is untouched.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rope_internal.h"

namespace rope {

// Programmatic dependent launch.  Every launch carries the programmatic
// stream-serialisation attribute, so the next kernel in the stream may start
// before this one has finished.  Each block first lets the next grid launch
// (it launches once every block of this grid has started, so its blocks
// never take the slots of blocks of ours that still wait to run), then
// waits until the grids it depends on have completed and their writes are
// visible.  No global memory is touched before that wait, so a call behaves
// exactly as if fully serialised after whatever the stream ran before it; what
// overlaps is only the launch and ramp of one grid with the tail of the
// previous one.  Without a programmatic predecessor the wait returns at once.
__device__ __forceinline__ void enter_after_predecessor() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int W>
struct Words {
    uint32_t w[W];
};

// ------------------------------------------------------------------------
// storage packing: pairs <-> 32-bit words
// ------------------------------------------------------------------------

template <typename T>
struct Pack;

template <>
struct Pack<float> {
    static constexpr int kWordsPerPair = 2;
    static __device__ __forceinline__ void get(const uint32_t* w, float& a, float& b) {
        a = __uint_as_float(w[0]);
        b = __uint_as_float(w[1]);
    }
    static __device__ __forceinline__ void put(uint32_t* w, float a, float b) {
        w[0] = __float_as_uint(a);
        w[1] = __float_as_uint(b);
    }
};

template <>
struct Pack<__nv_bfloat16> {
    static constexpr int kWordsPerPair = 1;
    // a bfloat16 is the top half of a binary32: widening is a shift
    static __device__ __forceinline__ void get(const uint32_t* w, float& a, float& b) {
        a = __uint_as_float(w[0] << 16);
        b = __uint_as_float(w[0] & 0xffff0000u);
    }
    static __device__ __forceinline__ void put(uint32_t* w, float a, float b) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x (low half) = a
        uint32_t u;
        memcpy(&u, &h, 4);
        w[0] = u;
    }
};

template <>
struct Pack<__half> {
    static constexpr int kWordsPerPair = 1;
    static __device__ __forceinline__ void get(const uint32_t* w, float& a, float& b) {
        __half2 h;
        memcpy(&h, &w[0], 4);
        const float2 f = __half22float2(h);
        a = f.x;
        b = f.y;
    }
    static __device__ __forceinline__ void put(uint32_t* w, float a, float b) {
        const __half2 h = __floats2half2_rn(a, b);  // .x (low half) = a
        uint32_t u;
        memcpy(&u, &h, 4);
        w[0] = u;
    }
};

// ------------------------------------------------------------------------
// global memory: x (read then written by the same thread) and cos/sin
// (read-only for the whole kernel, so they may take the non-coherent path)
// ------------------------------------------------------------------------

// x loads carry an explicit 64-byte L2 prefetch size.  Without it a miss
// pulls the whole 128-byte line from HBM; a slice that ends a few bytes into
// a line (e.g. bytes [136, 392) of a 512-byte row) then reads up to 120
// bytes it never uses.  64 bytes is the HBM access atom, so nothing smaller
// can be fetched anyway.  The asm is volatile so the U loads keep their
// order; each store depends on its own load's data, which orders them.
template <int W>
__device__ __forceinline__ Words<W> ld_vec(const char* p) {
    Words<W> v;
    if constexpr (W == 4) {
        asm volatile("ld.global.L2::64B.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                     : "l"(p));
    } else if constexpr (W == 2) {
        asm volatile("ld.global.L2::64B.v2.u32 {%0, %1}, [%2];"
                     : "=r"(v.w[0]), "=r"(v.w[1])
                     : "l"(p));
    } else {
        asm volatile("ld.global.L2::64B.u32 %0, [%1];" : "=r"(v.w[0]) : "l"(p));
    }
    return v;
}

template <int W>
__device__ __forceinline__ Words<W> ldg_vec(const char* p) {
    Words<W> v;
    if constexpr (W == 4) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
        v.w[0] = q.x; v.w[1] = q.y; v.w[2] = q.z; v.w[3] = q.w;
    } else if constexpr (W == 2) {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
        v.w[0] = q.x; v.w[1] = q.y;
    } else {
        v.w[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
    }
    return v;
}

template <int W>
__device__ __forceinline__ void st_vec(char* p, const Words<W>& v) {
    if constexpr (W == 4) {
        *reinterpret_cast<uint4*>(p) = make_uint4(v.w[0], v.w[1], v.w[2], v.w[3]);
    } else if constexpr (W == 2) {
        *reinterpret_cast<uint2*>(p) = make_uint2(v.w[0], v.w[1]);
    } else {
        *reinterpret_cast<uint32_t*>(p) = v.w[0];
    }
}

// One pair through element-sized accesses (any element-aligned address).
template <typename T, bool RO>
__device__ __forceinline__ Words<Pack<T>::kWordsPerPair> ld_pair_scalar(const char* p) {
    Words<Pack<T>::kWordsPerPair> v;
    if constexpr (sizeof(T) == 4) {
        const unsigned int* q = reinterpret_cast<const unsigned int*>(p);
        v.w[0] = RO ? __ldg(q) : q[0];
        v.w[1] = RO ? __ldg(q + 1) : q[1];
    } else {
        const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
        const uint32_t lo = RO ? __ldg(q) : q[0];
        const uint32_t hi = RO ? __ldg(q + 1) : q[1];
        v.w[0] = lo | (hi << 16);
    }
    return v;
}

template <typename T>
__device__ __forceinline__ void st_pair_scalar(char* p, const Words<Pack<T>::kWordsPerPair>& v) {
    if constexpr (sizeof(T) == 4) {
        unsigned int* q = reinterpret_cast<unsigned int*>(p);
        q[0] = v.w[0];
        q[1] = v.w[1];
    } else {
        unsigned short* q = reinterpret_cast<unsigned short*>(p);
        q[0] = static_cast<unsigned short>(v.w[0] & 0xffffu);
        q[1] = static_cast<unsigned short>(v.w[0] >> 16);
    }
}

// One element through an element-sized access, in the low bits of a word
// (the half-split mode's scalar path, where a pair's lanes are L/2 apart).
template <typename T, bool RO>
__device__ __forceinline__ Words<1> ld_elem_scalar(const char* p) {
    Words<1> v;
    if constexpr (sizeof(T) == 4) {
        const unsigned int* q = reinterpret_cast<const unsigned int*>(p);
        v.w[0] = RO ? __ldg(q) : q[0];
    } else {
        const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
        v.w[0] = RO ? __ldg(q) : q[0];
    }
    return v;
}

template <typename T>
__device__ __forceinline__ void st_elem_scalar(char* p, const Words<1>& v) {
    if constexpr (sizeof(T) == 4) *reinterpret_cast<unsigned int*>(p) = v.w[0];
    else *reinterpret_cast<unsigned short*>(p) = static_cast<unsigned short>(v.w[0] & 0xffffu);
}

// One element held in the low bits of a word.
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static __device__ __forceinline__ float get(uint32_t w) { return __uint_as_float(w); }
    static __device__ __forceinline__ uint32_t put(float v) { return __float_as_uint(v); }
};

template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float get(uint32_t w) { return __uint_as_float(w << 16); }
    static __device__ __forceinline__ uint32_t put(float v) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
};

template <>
struct Elem<__half> {
    static __device__ __forceinline__ float get(uint32_t w) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
    }
    static __device__ __forceinline__ uint32_t put(float v) {
        return __half_as_ushort(__float2half_rn(v));
    }
};

template <typename T, int W, bool SCALAR>
__device__ __forceinline__ Words<W> load_x(const char* p) {
    if constexpr (SCALAR) return ld_pair_scalar<T, false>(p);
    else return ld_vec<W>(p);
}

template <typename T, int W, bool SCALAR>
__device__ __forceinline__ Words<W> load_r(const char* p) {
    if constexpr (SCALAR) return ld_pair_scalar<T, true>(p);
    else return ldg_vec<W>(p);
}

template <typename T, int W, bool SCALAR>
__device__ __forceinline__ void store_x(char* p, const Words<W>& v) {
    if constexpr (SCALAR) st_pair_scalar<T>(p, v);
    else st_vec<W>(p, v);
}

// Accesses of the half-split mode: vector chunks as in interleave mode, or
// one element per access on the scalar path.
template <typename T, int W, bool SCALAR>
__device__ __forceinline__ Words<W> load_x_half(const char* p) {
    if constexpr (SCALAR) return ld_elem_scalar<T, false>(p);
    else return ld_vec<W>(p);
}

template <typename T, int W, bool SCALAR>
__device__ __forceinline__ Words<W> load_r_half(const char* p) {
    if constexpr (SCALAR) return ld_elem_scalar<T, true>(p);
    else return ldg_vec<W>(p);
}

template <typename T, int W, bool SCALAR>
__device__ __forceinline__ void store_x_half(char* p, const Words<W>& v) {
    if constexpr (SCALAR) st_elem_scalar<T>(p, v);
    else st_vec<W>(p, v);
}

// ------------------------------------------------------------------------
// the rotation of one pair, in the page's rounding order
// ------------------------------------------------------------------------

template <int DIR>
__device__ __forceinline__ void rotate_pair(float x0, float x1, float c0, float c1, float s0,
                                            float s1, float& y0, float& y1) {
    if constexpr (DIR == kFwd) {
        y0 = __fsub_rn(__fmul_rn(x0, c0), __fmul_rn(x1, s0));
        y1 = __fadd_rn(__fmul_rn(x1, c1), __fmul_rn(x0, s1));
    } else {
        y0 = __fadd_rn(__fmul_rn(x0, c0), __fmul_rn(x1, s1));
        y1 = __fsub_rn(__fmul_rn(x1, c1), __fmul_rn(x0, s0));
    }
}

template <typename T, int W, int DIR>
__device__ __forceinline__ Words<W> rotate_chunk(const Words<W>& x, const Words<W>& c,
                                                 const Words<W>& s) {
    using P = Pack<T>;
    constexpr int WPP = P::kWordsPerPair;
    Words<W> y;
#pragma unroll
    for (int p = 0; p < W / WPP; ++p) {
        float x0, x1, c0, c1, s0, s1, y0, y1;
        P::get(&x.w[p * WPP], x0, x1);
        P::get(&c.w[p * WPP], c0, c1);
        P::get(&s.w[p * WPP], s0, s1);
        rotate_pair<DIR>(x0, x1, c0, c1, s0, s1, y0, y1);
        P::put(&y.w[p * WPP], y0, y1);
    }
    return y;
}

// Half-split mode: element k of chunk A (lane j) pairs with element k of
// chunk B (lane j + L/2); cos/sin come from the same two lanes.
template <typename T, int W, bool SCALAR, int DIR>
__device__ __forceinline__ void rotate_half_chunks(const Words<W>& xa, const Words<W>& xb,
                                                   const Words<W>& ca, const Words<W>& cb,
                                                   const Words<W>& sa, const Words<W>& sb,
                                                   Words<W>& ya, Words<W>& yb) {
    if constexpr (SCALAR || sizeof(T) == 4) {
        // one element per word
#pragma unroll
        for (int w = 0; w < W; ++w) {
            float y0, y1;
            rotate_pair<DIR>(Elem<T>::get(xa.w[w]), Elem<T>::get(xb.w[w]), Elem<T>::get(ca.w[w]),
                             Elem<T>::get(cb.w[w]), Elem<T>::get(sa.w[w]), Elem<T>::get(sb.w[w]),
                             y0, y1);
            ya.w[w] = Elem<T>::put(y0);
            yb.w[w] = Elem<T>::put(y1);
        }
    } else {
        // two 16-bit elements per word
        using P = Pack<T>;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            float a0, a1, b0, b1, c0a, c1a, c0b, c1b, s0a, s1a, s0b, s1b;
            float ya0, ya1, yb0, yb1;
            P::get(&xa.w[w], a0, a1);
            P::get(&xb.w[w], b0, b1);
            P::get(&ca.w[w], c0a, c1a);
            P::get(&cb.w[w], c0b, c1b);
            P::get(&sa.w[w], s0a, s1a);
            P::get(&sb.w[w], s0b, s1b);
            rotate_pair<DIR>(a0, b0, c0a, c0b, s0a, s0b, ya0, yb0);
            rotate_pair<DIR>(a1, b1, c1a, c1b, s1a, s1b, ya1, yb1);
            P::put(&ya.w[w], ya0, ya1);
            P::put(&yb.w[w], yb0, yb1);
        }
    }
}

// ------------------------------------------------------------------------
// the kernel body
//   T      storage type            VEC    bytes per access of x
//   SCALAR element-wise accesses   U      heads per thread
//   DIR    kFwd / kBwd             RHEAD  cos/sin differ between heads
//   TWO    two tensors in one launch (the fused query + key call): the work
//          items of the first (x, N1 heads, H head groups) come first, those
//          of the second (x2, N - N1 heads, H2 head groups) after them, so
//          each tensor is swept in address order as a launch of its own
//          would; both use the token's one cos/sin row
//   HALF   half-split mode: the chunk covers lanes of the slice's first half
//          and pairs with the chunk half_off bytes further on (x and cos/sin)
// ------------------------------------------------------------------------

template <typename T, int VEC, bool SCALAR, int U, int DIR, bool RHEAD, bool TWO, bool HALF>
__device__ __forceinline__ void rope_body(const KernelArgs& a) {
    constexpr int W = VEC >= 4 ? VEC / 4 : 1;
    const char* const __restrict__ r1base = a.r1;
    const char* const __restrict__ r2base = a.r2;
    const uint64_t stride = uint64_t(gridDim.x) * kThreads;

    enter_after_predecessor();
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < a.tasks; t += stride) {
        uint32_t task = uint32_t(t), rest, c, tok, hg, b, s;
        char* xbase = a.x;
        int64_t tok_bytes = a.tok_bytes, row_bytes = a.row_bytes;
        int nheads = a.N;
        FastDiv divH = a.divH;
        if constexpr (TWO) {
            const bool second = task >= a.tasks1;
            if (second) task -= a.tasks1;
            xbase = second ? a.x2 : a.x;
            tok_bytes = second ? a.tok_bytes2 : a.tok_bytes;
            row_bytes = second ? a.row_bytes2 : a.row_bytes;
            nheads = second ? a.N - a.N1 : a.N1;
            divH = second ? a.divH2 : a.divH;
        }
        a.divC.divmod(task, rest, c);
        divH.divmod(rest, tok, hg);
        a.divS.divmod(tok, b, s);

        // this thread's heads are n0 .. n0 + U - 1 (consecutive rows)
        const int n0 = int(hg) * U;
        const int64_t c_off = int64_t(c) * VEC;
        char* xp[U];
        {
            char* x0 = xbase + int64_t(tok) * tok_bytes + int64_t(n0) * row_bytes + c_off;
#pragma unroll
            for (int i = 0; i < U; ++i) xp[i] = x0 + i * row_bytes;
        }
        const char* c_p = r1base + int64_t(b) * a.r1_b + int64_t(s) * a.r1_s + c_off;
        const char* s_p = r2base + int64_t(b) * a.r2_b + int64_t(s) * a.r2_s + c_off;
        if constexpr (RHEAD) {
            c_p += int64_t(n0) * a.r1_n;
            s_p += int64_t(n0) * a.r2_n;
        }

        if constexpr (HALF) {
            const int64_t ho = a.half_off;
            Words<W> xa[U], xb[U];
#pragma unroll
            for (int i = 0; i < U; ++i)
                if (i == 0 || n0 + i < nheads) {
                    xa[i] = load_x_half<T, W, SCALAR>(xp[i]);
                    xb[i] = load_x_half<T, W, SCALAR>(xp[i] + ho);
                }
            Words<W> ca, cb, sa, sb;
            if constexpr (!RHEAD) {
                ca = load_r_half<T, W, SCALAR>(c_p);
                cb = load_r_half<T, W, SCALAR>(c_p + ho);
                sa = load_r_half<T, W, SCALAR>(s_p);
                sb = load_r_half<T, W, SCALAR>(s_p + ho);
            }
#pragma unroll
            for (int i = 0; i < U; ++i) {
                if (i == 0 || n0 + i < nheads) {
                    if constexpr (RHEAD) {
                        const int64_t o1 = int64_t(i) * a.r1_n, o2 = int64_t(i) * a.r2_n;
                        ca = load_r_half<T, W, SCALAR>(c_p + o1);
                        cb = load_r_half<T, W, SCALAR>(c_p + o1 + ho);
                        sa = load_r_half<T, W, SCALAR>(s_p + o2);
                        sb = load_r_half<T, W, SCALAR>(s_p + o2 + ho);
                    }
                    Words<W> ya, yb;
                    rotate_half_chunks<T, W, SCALAR, DIR>(xa[i], xb[i], ca, cb, sa, sb, ya, yb);
                    store_x_half<T, W, SCALAR>(xp[i], ya);
                    store_x_half<T, W, SCALAR>(xp[i] + ho, yb);
                }
            }
            continue;
        }

        Words<W> xv[U];
#pragma unroll
        for (int i = 0; i < U; ++i)
            if (i == 0 || n0 + i < nheads) xv[i] = load_x<T, W, SCALAR>(xp[i]);

        Words<W> cv, sv;
        if constexpr (!RHEAD) {
            cv = load_r<T, W, SCALAR>(c_p);
            sv = load_r<T, W, SCALAR>(s_p);
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (i == 0 || n0 + i < nheads) {
                if constexpr (RHEAD) {
                    cv = load_r<T, W, SCALAR>(c_p + int64_t(i) * a.r1_n);
                    sv = load_r<T, W, SCALAR>(s_p + int64_t(i) * a.r2_n);
                }
                store_x<T, W, SCALAR>(xp[i], rotate_chunk<T, W, DIR>(xv[i], cv, sv));
            }
        }
    }
}

// One tensor.
template <typename T, int VEC, bool SCALAR, int U, int DIR, bool RHEAD>
__global__ void __launch_bounds__(kThreads) rope_partial_kernel(const KernelArgs a) {
    rope_body<T, VEC, SCALAR, U, DIR, RHEAD, false, false>(a);
}

// Query and key in one launch, sharing each token's cos/sin row.
template <typename T, int VEC, bool SCALAR, int U, int DIR>
__global__ void __launch_bounds__(kThreads) rope_partial_qk_kernel(const KernelArgs a) {
    rope_body<T, VEC, SCALAR, U, DIR, false, true, false>(a);
}

// One tensor, half-split mode (pairs (j, j + L/2)).
template <typename T, int VEC, bool SCALAR, int U, int DIR, bool RHEAD>
__global__ void __launch_bounds__(kThreads) rope_partial_half_kernel(const KernelArgs a) {
    rope_body<T, VEC, SCALAR, U, DIR, RHEAD, false, true>(a);
}

// ------------------------------------------------------------------------
// 16-bit interleave mode with an odd start: pairs across aligned words
// ------------------------------------------------------------------------
// With an odd start, pair p of a row (elements start + 2p and start + 2p + 1)
// straddles two aligned 4-byte words: the high half of word p and the low
// half of word p + 1, counting words from the one that holds element
// start - 1.  For rows of P pairs with P a power of two in [1, 32], lane p
// of a row loads word p (a warp's loads are contiguous), takes the low half
// of word p + 1 from lane p + 1 by shuffle (the row's last lane loads word P
// itself) and stores word p whole: its low half is the previous pair's
// second result, taken from lane p - 1 by shuffle.  The row's first lane
// stores only the high half of word 0 and its last lane only the low half of
// word P (2-byte stores), so no byte outside the slice is written.
template <typename T, int U, int DIR, bool RHEAD>
__global__ void __launch_bounds__(kThreads) rope_partial_odd_kernel(const KernelArgs a) {
    static_assert(sizeof(T) == 2, "the odd-start path is for 16-bit storage");
    using P = Pack<T>;
    const uint32_t C = a.divC.d;  // pairs (= lanes) per row: a power of two in [1, 32]
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t stride = uint64_t(gridDim.x) * kThreads;
    enter_after_predecessor();
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < a.tasks; t += stride) {
        // the lanes of this warp still in the loop (tasks is a multiple of C,
        // so they hold whole rows)
        const uint64_t left = a.tasks - (t - lane);
        const uint32_t mask = left >= 32 ? 0xffffffffu : ((1u << uint32_t(left)) - 1u);
        uint32_t rest, p, tok, hg, b, s;
        a.divC.divmod(uint32_t(t), rest, p);
        a.divH.divmod(rest, tok, hg);
        a.divS.divmod(tok, b, s);
        const bool first = p == 0, last = p + 1 == C;
        const int n0 = int(hg) * U;
        // word p of head n0's row: row elements start - 1 + 2p (low half)
        // and start + 2p (high half)
        char* w0 = a.x - 2 + int64_t(tok) * a.tok_bytes + int64_t(n0) * a.row_bytes + int64_t(p) * 4;
        const char* c_p = a.r1 + int64_t(b) * a.r1_b + int64_t(s) * a.r1_s + int64_t(p) * 4;
        const char* s_p = a.r2 + int64_t(b) * a.r2_b + int64_t(s) * a.r2_s + int64_t(p) * 4;
        if constexpr (RHEAD) {
            c_p += int64_t(n0) * a.r1_n;
            s_p += int64_t(n0) * a.r2_n;
        }

        uint32_t xw[U], xn[U];  // word p, and word p + 1 for the row's last lane
#pragma unroll
        for (int i = 0; i < U; ++i) {
            xw[i] = 0u;
            xn[i] = 0u;
            if (i == 0 || n0 + i < a.N) {
                xw[i] = ld_vec<1>(w0 + i * a.row_bytes).w[0];
                if (last) xn[i] = ld_vec<1>(w0 + i * a.row_bytes + 4).w[0];
            }
        }
        uint32_t cw = 0u, sw = 0u;
        if constexpr (!RHEAD) {
            cw = ldg_vec<1>(c_p).w[0];
            sw = ldg_vec<1>(s_p).w[0];
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            // every lane of `mask` shuffles, outside any per-lane condition
            const uint32_t down = __shfl_down_sync(mask, xw[i], 1);
            const uint32_t nxt = last ? xn[i] : down;
            if constexpr (RHEAD) {
                if (i == 0 || n0 + i < a.N) {
                    cw = ldg_vec<1>(c_p + int64_t(i) * a.r1_n).w[0];
                    sw = ldg_vec<1>(s_p + int64_t(i) * a.r2_n).w[0];
                }
            }
            float lo, x0, x1, hi, c0, c1, s0, s1, y0, y1;
            P::get(&xw[i], lo, x0);  // x0: element start + 2p
            P::get(&nxt, x1, hi);    // x1: element start + 2p + 1
            P::get(&cw, c0, c1);
            P::get(&sw, s0, s1);
            rotate_pair<DIR>(x0, x1, c0, c1, s0, s1, y0, y1);
            const uint32_t y0b = Elem<T>::put(y0), y1b = Elem<T>::put(y1);
            const uint32_t prev = __shfl_up_sync(mask, y1b, 1);  // the previous pair's second result
            if (i == 0 || n0 + i < a.N) {
                char* wp = w0 + i * a.row_bytes;
                if (first) {
                    st_elem_scalar<T>(wp + 2, Words<1>{{y0b}});
                } else {
                    st_vec<1>(wp, Words<1>{{(prev & 0xffffu) | (y0b << 16)}});
                }
                if (last) st_elem_scalar<T>(wp + 4, Words<1>{{y1b}});
            }
        }
    }
}

// ------------------------------------------------------------------------
// half-split mode with the partner access in another lane
// ------------------------------------------------------------------------
// When a row's slice is C accesses long with C a power of two in [2, 32],
// the work index puts the row's C accesses in C consecutive lanes of one
// warp (C divides 32, so rows never straddle warps), and the access that
// holds lane j + L/2 is the one C/2 lanes on.  Each thread then loads only
// its own access of x, cos and sin, exactly as in interleave mode, and takes
// the partner's x (and, in the backward, the partner's sin) with one warp
// shuffle per 32-bit word.  Against pairing two accesses in one thread this
// halves the registers per thread and lets 8 lanes cover a whole 128-byte
// line of the slice.

// One lane of a half-split pair, in the rounding order of rotate_pair.  For
// the first-half lane j (own = x_j, other = x_{j+L/2}) and the second-half
// lane j + L/2 (own = x_{j+L/2}, other = x_j), with c, s the own lane's
// cos/sin and s_other the partner lane's sin:
//   forward : first  own*c - other*s        second  own*c + other*s
//   backward: first  own*c + other*s_other  second  own*c - other*s_other
// Each is own*c + (±other)*s': the sign goes onto `other` before the
// multiply (flipping sign bits is exact, fl(-a*b) = -fl(a*b), and a - b is
// a + (-b) in IEEE arithmetic), so a lane costs what an interleaved pair
// does: two products and one sum per element, plus one XOR per word.
template <typename T, int W, int DIR>
__device__ __forceinline__ Words<W> rotate_chunk_lanes(bool first, const Words<W>& x,
                                                       const Words<W>& xo, const Words<W>& c,
                                                       const Words<W>& s, const Words<W>& so) {
    constexpr uint32_t kSign = sizeof(T) == 4 ? 0x80000000u : 0x80008000u;
    const uint32_t neg = (DIR == kFwd) == first ? kSign : 0u;
    const Words<W>& sx = DIR == kFwd ? s : so;
    Words<W> y;
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int w = 0; w < W; ++w)
            y.w[w] = __float_as_uint(__fadd_rn(
                __fmul_rn(__uint_as_float(x.w[w]), __uint_as_float(c.w[w])),
                __fmul_rn(__uint_as_float(xo.w[w] ^ neg), __uint_as_float(sx.w[w]))));
    } else {
        // element k of a word pairs with element k of the partner's word
        using P = Pack<T>;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const uint32_t o = xo.w[w] ^ neg;
            float x0, x1, o0, o1, c0, c1, s0, s1;
            P::get(&x.w[w], x0, x1);
            P::get(&o, o0, o1);
            P::get(&c.w[w], c0, c1);
            P::get(&sx.w[w], s0, s1);
            P::put(&y.w[w], __fadd_rn(__fmul_rn(x0, c0), __fmul_rn(o0, s0)),
                   __fadd_rn(__fmul_rn(x1, c1), __fmul_rn(o1, s1)));
        }
    }
    return y;
}

template <int W>
__device__ __forceinline__ Words<W> shfl_xor_words(uint32_t mask, const Words<W>& v, int lanes) {
    Words<W> o;
#pragma unroll
    for (int w = 0; w < W; ++w) o.w[w] = __shfl_xor_sync(mask, v.w[w], lanes);
    return o;
}

// One tensor, half-split mode, partner access in lane ^ C/2.
template <typename T, int VEC, int U, int DIR, bool RHEAD>
__global__ void __launch_bounds__(kThreads) rope_partial_half_lanes_kernel(const KernelArgs a) {
    constexpr int W = VEC / 4;
    constexpr int R = RHEAD ? U : 1;  // cos/sin accesses per thread
    const uint32_t C = a.divC.d;      // accesses per row: a power of two in [2, 32]
    const int other = int(C >> 1);    // lane distance to the partner access
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t stride = uint64_t(gridDim.x) * kThreads;

    enter_after_predecessor();
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < a.tasks; t += stride) {
        // the lanes of this warp still in the loop: items t - lane .. tasks - 1
        // (tasks is a multiple of C, so a lane's partner is always among them)
        const uint64_t left = a.tasks - (t - lane);
        const uint32_t mask = left >= 32 ? 0xffffffffu : ((1u << uint32_t(left)) - 1u);
        uint32_t rest, c, tok, hg, b, s;
        a.divC.divmod(uint32_t(t), rest, c);
        a.divH.divmod(rest, tok, hg);
        a.divS.divmod(tok, b, s);
        const bool first = c < C / 2;
        const int n0 = int(hg) * U;
        const int64_t c_off = int64_t(c) * VEC;
        char* x0 = a.x + int64_t(tok) * a.tok_bytes + int64_t(n0) * a.row_bytes + c_off;
        const char* c_p = a.r1 + int64_t(b) * a.r1_b + int64_t(s) * a.r1_s + c_off;
        const char* s_p = a.r2 + int64_t(b) * a.r2_b + int64_t(s) * a.r2_s + c_off;
        if constexpr (RHEAD) {
            c_p += int64_t(n0) * a.r1_n;
            s_p += int64_t(n0) * a.r2_n;
        }

        // loads (heads past N read nothing and hold zeros)
        Words<W> xv[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (i == 0 || n0 + i < a.N) xv[i] = load_x<T, W, false>(x0 + i * a.row_bytes);
            else xv[i] = Words<W>{};
        }
        Words<W> cv[R], sv[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            if (j == 0 || n0 + j < a.N) {
                cv[j] = load_r<T, W, false>(c_p + int64_t(j) * a.r1_n);
                sv[j] = load_r<T, W, false>(s_p + int64_t(j) * a.r2_n);
            } else {
                cv[j] = Words<W>{};
                sv[j] = Words<W>{};
            }
        }
        // the partner's values: every lane of `mask` shuffles, outside any
        // per-lane condition
        Words<W> so[R];
#pragma unroll
        for (int j = 0; j < R; ++j) so[j] = DIR == kBwd ? shfl_xor_words<W>(mask, sv[j], other) : sv[j];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const Words<W> xo = shfl_xor_words<W>(mask, xv[i], other);
            if (i == 0 || n0 + i < a.N) {
                const int j = RHEAD ? i : 0;
                store_x<T, W, false>(x0 + i * a.row_bytes,
                                     rotate_chunk_lanes<T, W, DIR>(first, xv[i], xo, cv[j], sv[j], so[j]));
            }
        }
    }
}

// ------------------------------------------------------------------------
// cos/sin computed from positions (no table read)
// ------------------------------------------------------------------------

// 2*pi as three fp32 parts, each the fp32 rounding of what the parts before
// it leave of 2*pi = 6.28318530717958647692528676655900576839... (remainder
// after the three: 4.2e-23).  The first part's 24-bit significand makes
// n * A exact inside an FMA for every |n| < 2^22.
__device__ __forceinline__ float two_pi_a() { return __uint_as_float(0x40c90fdbu); }  //  6.2831855
__device__ __forceinline__ float two_pi_b() { return __uint_as_float(0xb43bbd2eu); }  // -1.7484555e-07
__device__ __forceinline__ float two_pi_c() { return __uint_as_float(0xa7f72cedu); }  // -6.8604980e-15
__device__ __forceinline__ float inv_two_pi() { return __uint_as_float(0x3e22f983u); } //  0.15915494

// cos and sin of theta = p * omega, omega = hi + lo.  theta is carried as
// th + tl (th = p*hi rounded; tl = the exact residual of that product plus
// p*lo), so it is accurate to about 2^-44 relative for |p| < 2^24 (p is
// then exact in fp32).  Reduction by 2*pi follows Cody and Waite
// ("Software Manual for the Elementary Functions", 1980) with the three-part
// constant above: r = ((th - n*A) - n*B) - n*C + tl, where the first step is
// exact (Sterbenz when |th| < 4, otherwise both terms are multiples of the
// first part's ulp and the difference has at most 23 bits).  The other three
// steps round once each, so |r - (theta - 2*pi*n)| <= 3 * 2^-23 and |r| stays
// within pi plus a rounding.  On that range the hardware __sincosf has an
// absolute error of at most 2^-21.41 (CUDA's documented bound for |x| <= pi),
// so the cos/sin used are within 2^-21.41 + 3 * 2^-23 < 8e-7 of the exact
// values, at a few instructions per angle.
__device__ __forceinline__ void angle_cos_sin(float p, float w_hi, float w_lo, float& c, float& s) {
    const float th = __fmul_rn(p, w_hi);
    const float tl = __fmaf_rn(p, w_lo, __fmaf_rn(p, w_hi, -th));
    const float n = rintf(__fmul_rn(th, inv_two_pi()));
    float r = __fmaf_rn(-n, two_pi_a(), th);
    r = __fmaf_rn(-n, two_pi_b(), r);
    r = __fmaf_rn(-n, two_pi_c(), r);
    r = __fadd_rn(r, tl);
    __sincosf(r, &s, &c);
}

// Interleave mode: pair j of the chunk uses angle j.
template <typename T, int W, int DIR>
__device__ __forceinline__ Words<W> rotate_chunk_angles(const Words<W>& x, const float* cs,
                                                        const float* sn) {
    using P = Pack<T>;
    constexpr int WPP = P::kWordsPerPair;
    Words<W> y;
#pragma unroll
    for (int p = 0; p < W / WPP; ++p) {
        float x0, x1, y0, y1;
        P::get(&x.w[p * WPP], x0, x1);
        rotate_pair<DIR>(x0, x1, cs[p], cs[p], sn[p], sn[p], y0, y1);
        P::put(&y.w[p * WPP], y0, y1);
    }
    return y;
}

// Half-split mode: element k of chunk A and of chunk B use angle k.
template <typename T, int W, bool SCALAR, int DIR>
__device__ __forceinline__ void rotate_half_angles(const Words<W>& xa, const Words<W>& xb,
                                                   const float* cs, const float* sn,
                                                   Words<W>& ya, Words<W>& yb) {
    if constexpr (SCALAR || sizeof(T) == 4) {
#pragma unroll
        for (int w = 0; w < W; ++w) {
            float y0, y1;
            rotate_pair<DIR>(Elem<T>::get(xa.w[w]), Elem<T>::get(xb.w[w]), cs[w], cs[w], sn[w],
                             sn[w], y0, y1);
            ya.w[w] = Elem<T>::put(y0);
            yb.w[w] = Elem<T>::put(y1);
        }
    } else {
        using P = Pack<T>;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            float a0, a1, b0, b1, ya0, ya1, yb0, yb1;
            P::get(&xa.w[w], a0, a1);
            P::get(&xb.w[w], b0, b1);
            rotate_pair<DIR>(a0, b0, cs[2 * w], cs[2 * w], sn[2 * w], sn[2 * w], ya0, yb0);
            rotate_pair<DIR>(a1, b1, cs[2 * w + 1], cs[2 * w + 1], sn[2 * w + 1], sn[2 * w + 1],
                             ya1, yb1);
            P::put(&ya.w[w], ya0, ya1);
            P::put(&yb.w[w], yb0, yb1);
        }
    }
}

// The positions call: the task loop of rope_body with each chunk's cos/sin
// computed once per thread (shared by its U heads) instead of loaded.
template <typename T, int VEC, bool SCALAR, int U, int DIR, bool HALF>
__global__ void __launch_bounds__(kThreads)
rope_partial_pos_kernel(const KernelArgs a, const FreqTable f) {
    __shared__ float w_hi[kMaxPairs];
    __shared__ float w_lo[kMaxPairs];
    for (int i = threadIdx.x; i < a.pairs; i += kThreads) {
        w_hi[i] = f.hi[i];
        w_lo[i] = f.lo[i];
    }
    __syncthreads();

    constexpr int W = VEC >= 4 ? VEC / 4 : 1;
    constexpr int E = VEC / int(sizeof(T)) > 0 ? VEC / int(sizeof(T)) : 1;  // elements per chunk
    // angles per chunk: half-split one per element; interleave one per pair
    constexpr int NA = HALF ? E : (E / 2 > 0 ? E / 2 : 1);
    const uint64_t stride = uint64_t(gridDim.x) * kThreads;

    enter_after_predecessor();
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < a.tasks; t += stride) {
        uint32_t rest, c, tok, hg, b, s;
        a.divC.divmod(uint32_t(t), rest, c);
        a.divH.divmod(rest, tok, hg);
        a.divS.divmod(tok, b, s);
        const int n0 = int(hg) * U;
        char* x0 = a.x + int64_t(tok) * a.tok_bytes + int64_t(n0) * a.row_bytes + int64_t(c) * VEC;

        Words<W> xa[U], xb[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (i == 0 || n0 + i < a.N) {
                if constexpr (HALF) {
                    xa[i] = load_x_half<T, W, SCALAR>(x0 + i * a.row_bytes);
                    xb[i] = load_x_half<T, W, SCALAR>(x0 + i * a.row_bytes + a.half_off);
                } else {
                    xa[i] = load_x<T, W, SCALAR>(x0 + i * a.row_bytes);
                }
            }
        }

        const float p = __int2float_rn(__ldg(a.pos + int64_t(b) * a.pos_b + int64_t(s) * a.pos_s));
        const int k0 = int(c) * NA;
        float cs[NA], sn[NA];
#pragma unroll
        for (int j = 0; j < NA; ++j) angle_cos_sin(p, w_hi[k0 + j], w_lo[k0 + j], cs[j], sn[j]);

#pragma unroll
        for (int i = 0; i < U; ++i) {
            if (i == 0 || n0 + i < a.N) {
                char* xp = x0 + i * a.row_bytes;
                if constexpr (HALF) {
                    Words<W> ya, yb;
                    rotate_half_angles<T, W, SCALAR, DIR>(xa[i], xb[i], cs, sn, ya, yb);
                    store_x_half<T, W, SCALAR>(xp, ya);
                    store_x_half<T, W, SCALAR>(xp + a.half_off, yb);
                } else {
                    store_x<T, W, SCALAR>(xp, rotate_chunk_angles<T, W, DIR>(xa[i], cs, sn));
                }
            }
        }
    }
}

// ------------------------------------------------------------------------
// kernel selection for one storage type (instantiated in one .cu per type)
// ------------------------------------------------------------------------

enum Kind { kSingle, kQK, kHalfSplit, kHalfLanes, kPos, kPosHalf, kOdd };

template <typename T, int VEC, bool SCALAR, int U, Kind K>
const void* pick_dir(const Plan& p) {
    const bool f = p.dir == kFwd;
    if constexpr (K == kPos || K == kPosHalf) {
        constexpr bool H = K == kPosHalf;
        return f ? reinterpret_cast<const void*>(&rope_partial_pos_kernel<T, VEC, SCALAR, U, kFwd, H>)
                 : reinterpret_cast<const void*>(&rope_partial_pos_kernel<T, VEC, SCALAR, U, kBwd, H>);
    } else if constexpr (K == kOdd) {
        if constexpr (sizeof(T) == 2) {
            if (f)
                return p.r_head ? reinterpret_cast<const void*>(&rope_partial_odd_kernel<T, U, kFwd, true>)
                                : reinterpret_cast<const void*>(&rope_partial_odd_kernel<T, U, kFwd, false>);
            return p.r_head ? reinterpret_cast<const void*>(&rope_partial_odd_kernel<T, U, kBwd, true>)
                            : reinterpret_cast<const void*>(&rope_partial_odd_kernel<T, U, kBwd, false>);
        } else {
            return nullptr;
        }
    } else if constexpr (K == kQK) {
        return f ? reinterpret_cast<const void*>(&rope_partial_qk_kernel<T, VEC, SCALAR, U, kFwd>)
                 : reinterpret_cast<const void*>(&rope_partial_qk_kernel<T, VEC, SCALAR, U, kBwd>);
    } else if constexpr (K == kHalfLanes) {
        if (f)
            return p.r_head ? reinterpret_cast<const void*>(&rope_partial_half_lanes_kernel<T, VEC, U, kFwd, true>)
                            : reinterpret_cast<const void*>(&rope_partial_half_lanes_kernel<T, VEC, U, kFwd, false>);
        return p.r_head ? reinterpret_cast<const void*>(&rope_partial_half_lanes_kernel<T, VEC, U, kBwd, true>)
                        : reinterpret_cast<const void*>(&rope_partial_half_lanes_kernel<T, VEC, U, kBwd, false>);
    } else if constexpr (K == kHalfSplit) {
        if (f)
            return p.r_head ? reinterpret_cast<const void*>(&rope_partial_half_kernel<T, VEC, SCALAR, U, kFwd, true>)
                            : reinterpret_cast<const void*>(&rope_partial_half_kernel<T, VEC, SCALAR, U, kFwd, false>);
        return p.r_head ? reinterpret_cast<const void*>(&rope_partial_half_kernel<T, VEC, SCALAR, U, kBwd, true>)
                        : reinterpret_cast<const void*>(&rope_partial_half_kernel<T, VEC, SCALAR, U, kBwd, false>);
    } else {
        if (f)
            return p.r_head ? reinterpret_cast<const void*>(&rope_partial_kernel<T, VEC, SCALAR, U, kFwd, true>)
                            : reinterpret_cast<const void*>(&rope_partial_kernel<T, VEC, SCALAR, U, kFwd, false>);
        return p.r_head ? reinterpret_cast<const void*>(&rope_partial_kernel<T, VEC, SCALAR, U, kBwd, true>)
                        : reinterpret_cast<const void*>(&rope_partial_kernel<T, VEC, SCALAR, U, kBwd, false>);
    }
}

template <typename T, int VEC, bool SCALAR, Kind K>
const void* pick_heads(const Plan& p) {
    switch (p.U) {
        case 1: return pick_dir<T, VEC, SCALAR, 1, K>(p);
        case 2: return pick_dir<T, VEC, SCALAR, 2, K>(p);
        case 4: return pick_dir<T, VEC, SCALAR, 4, K>(p);
        case 8:
            if constexpr (VEC < 16) return pick_dir<T, VEC, SCALAR, 8, K>(p);
            else return nullptr;
        default: return nullptr;
    }
}

// Interleave mode (single tensor or query + key): 16/8/4-byte chunks of
// whole pairs, or a pair through element accesses.
template <typename T, Kind K>
const void* pick_interleave(const Plan& p) {
    if (p.path == kScalarPair) return pick_heads<T, 2 * sizeof(T), true, K>(p);
    switch (p.vec) {
        case 16: return pick_heads<T, 16, false, K>(p);
        case 8: return pick_heads<T, 8, false, K>(p);
        case 4:
            if constexpr (sizeof(T) == 2) return pick_heads<T, 4, false, K>(p);
            else return nullptr;
        default: return nullptr;
    }
}

// Half-split mode with the partner access in another lane: 16/8/4-byte
// accesses.
template <typename T>
const void* pick_half_lanes(const Plan& p) {
    switch (p.vec) {
        case 16: return pick_heads<T, 16, false, kHalfLanes>(p);
        case 8: return pick_heads<T, 8, false, kHalfLanes>(p);
        case 4: return pick_heads<T, 4, false, kHalfLanes>(p);
        default: return nullptr;
    }
}

// Half-split mode: 16/8/4-byte chunks, or single 16-bit elements.
template <typename T, Kind K>
const void* pick_half(const Plan& p) {
    if (p.path == kScalarPair) {
        if constexpr (sizeof(T) == 2) return pick_heads<T, 2, true, K>(p);
        else return nullptr;  // an fp32 element is a 4-byte chunk
    }
    switch (p.vec) {
        case 16: return pick_heads<T, 16, false, K>(p);
        case 8: return pick_heads<T, 8, false, K>(p);
        case 4: return pick_heads<T, 4, false, K>(p);
        default: return nullptr;
    }
}

template <typename T>
const void* pick_kernel(const Plan& p) {
    if (p.path == kOddPair) {
        if constexpr (sizeof(T) == 2) return pick_heads<T, 4, false, kOdd>(p);
        else return nullptr;
    }
    if (p.pos) return p.half ? pick_half<T, kPosHalf>(p) : pick_interleave<T, kPos>(p);
    if (p.half) return p.lanes ? pick_half_lanes<T>(p) : pick_half<T, kHalfSplit>(p);
    if (p.two) return pick_interleave<T, kQK>(p);
    return pick_interleave<T, kSingle>(p);
}

// defined in rope_kernels_{bf16,fp16,fp32}.cu
const void* kernel_for_bf16(const Plan& p);
const void* kernel_for_fp16(const Plan& p);
const void* kernel_for_fp32(const Plan& p);

}  // namespace rope

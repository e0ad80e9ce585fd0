// rope_kernels.cuh -- the sm_103a kernels of the in-place partial rotary
// embedding, forward and backward, for bf16 / fp16 / fp32 storage:
//   rope_partial_kernel      one tensor, interleaved pairs (the page's mode)
//   rope_partial_half_kernel one tensor, half-split pairs (i, i + L/2)
//   rope_partial_half_lanes_kernel  the same when a row's accesses fit one
//                            warp: the partner access comes by warp shuffle
//   rope_partial_qk_kernel   query and key in one launch, one cos/sin row
//   rope_partial_pos_kernel  cos/sin computed from positions (no table)
//   rope_partial_odd_kernel  interleave with an odd start at element 1 of an
//                            aligned 16- or 8-byte vector: a lane per
//                            vector, the straddling elements by shuffle
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
//     same thread; with an odd start every pair straddles two aligned
//     accesses, and a slice that starts at element 1 of an aligned vector
//     takes a lane per vector with the straddling elements brought by
//     shuffle;
//   * a thread keeps the chunk's cos/sin in registers and walks U
//     consecutive heads of the same token (heads hg*U .. hg*U + U - 1),
//     issuing all U loads of x before any arithmetic, so U accesses per
//     thread are in flight and the cos/sin bytes are read once per U heads;
//   * consecutive threads take consecutive chunks of a row, so a warp reads
//     whole 32-byte sectors of each row's slice;
//   * the flat work index is split by three multiply-high divisions per
//     item; the grid covers it once (one block per 256 items, so the
//     hardware starts a block as each one ends), except for 16-bit rows read
//     over the host link, where a grid of the resident blocks of all SMs
//     strides over the work (the host picks; both measured);
//   * launches use programmatic dependent launch: every kernel waits on
//     griddepcontrol before its first global access, so only its launch and
//     ramp overlap the tail of the kernel before it in the stream.
// Only slice bytes are written; every other byte of x is left as it was.
// Reads stay inside each row: the odd-start kernel also reads the elements
// of its edge vectors outside the slice (at least element start - 1 and the
// word that holds element end); the other kernels read only slice bytes.
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
// global memory: x (each byte read and then written by the same thread,
// except in the odd-start kernel, whose lanes also read a neighbour's edge
// word that they never write) and cos/sin (read-only for the whole kernel,
// so they may take the non-coherent path)
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
        } else {
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
// interleave mode with an odd start: pairs straddle aligned accesses
// ------------------------------------------------------------------------
// With an odd start, the first element of every pair sits at an odd offset
// from any aligned access of x.  This kernel takes slices that start at
// element 1 of an aligned V-byte vector of the row (VE = V / e elements; V
// = 16 or 8).  Lane j of a row owns the row's j-th such vector counted from
// the one that holds element `start` (vector-relative element q = VE * j +
// i) and rotates the PV = VE / 2 pairs whose first element lies in it:
// pair m takes elements 2m + 1 and 2m + 2, so the last pair's second
// element is element 0 of the next vector, brought from the next lane by
// one shuffle.  The lane then stores its vector whole; its element 0 is the
// previous lane's last second result, brought by one more shuffle.  Lane
// j's pair m is slice pair w = PV * j + m (valid for w < P, the row's
// pairs), and its cos/sin are the pair-aligned elements 2w, 2w + 1 of its
// cos/sin row, V bytes per lane.
//
// Only a row's edge lanes store less: the first from element 1 (`start`)
// on, the last up to `end`, in the fewest aligned pieces (below), so no
// byte outside the slice is written; the last lane also stores element 0
// of the vector after its own when the slice ends there.  A row's lanes are
// consecutive work items, so a row may straddle two warps.  The pair that
// straddles them belongs wholly to lane 31: it loads the next vector's
// first word itself and stores that pair's second result there, as a row's
// last lane does, and lane 0 of the next warp leaves its element 0 alone.
// No lane reads an element that another lane writes, except through a
// shuffle, so the in-place update has no race.
//
// Reads: whole vectors, so a row's first lane also reads element start - 1
// and its last lane may read elements past the slice up to its vector's end,
// and the word that holds element `end` (which exists: end is odd, D even);
// none of them is written.
//
//   T   storage type    V    bytes per access of x (16 or 8)
//   U   heads per thread     DIR  kFwd / kBwd     RHEAD  cos/sin per head
// a.odd_wide (uniform) says the cos/sin rows are V-aligned, so a lane whose
// pairs are all in the slice loads them with one V-byte access; otherwise
// each pair's cos/sin is loaded by words.

// Cos (or sin) of lane pairs [0, m_hi) (pair m at word m * WPP); the others
// hold zero and nothing outside the row is read.
template <typename T, int V>
__device__ __forceinline__ Words<V / 4> load_lane_r(const char* row, int w0, int m_hi, bool wide) {
    constexpr int W = V / 4;
    constexpr int WPP = Pack<T>::kWordsPerPair;
    constexpr int PV = W / WPP;
    constexpr int PB = 2 * int(sizeof(T));  // bytes of one pair
    if (wide && m_hi == PV) return ldg_vec<W>(row + int64_t(w0) * PB);
    Words<W> r;
#pragma unroll
    for (int m = 0; m < PV; ++m) {
#pragma unroll
        for (int k = 0; k < WPP; ++k) {
            r.w[m * WPP + k] = 0u;
            if (m < m_hi)
                r.w[m * WPP + k] =
                    __ldg(reinterpret_cast<const unsigned int*>(row + int64_t(w0 + m) * PB + 4 * k));
        }
    }
    return r;
}

// First and second element of lane pair m from the vector's words xw[0..W)
// and the next vector's first word xw[W].
template <typename T, int W>
__device__ __forceinline__ void odd_pair_x(const uint32_t* xw, int m, float& x0, float& x1) {
    if constexpr (sizeof(T) == 2) {
        float lo, hi;
        Pack<T>::get(&xw[m], lo, hi);
        x0 = hi;  // element 2m + 1: high half of word m
        Pack<T>::get(&xw[m + 1], lo, hi);
        x1 = lo;  // element 2m + 2: low half of word m + 1
    } else {
        x0 = __uint_as_float(xw[2 * m + 1]);
        x1 = __uint_as_float(xw[2 * m + 2]);
    }
}

// Edge lanes of the odd-start kernel store part of their vector: elements
// [lo, hi), lo = 0 or 1, hi odd or the whole vector.  Within one launch every
// row's first lanes have the same range, and so do its last lanes, so a lane
// picks its range's store sequence by value and each sequence is fixed at
// compile time: a 2-byte store of a cut word's half at each end and the
// whole words between in the widest aligned pieces (16, 8, 4 bytes).
// That is the fewest stores (and L2 write requests) the range allows.  They
// are host functions too, so that a host program can check every range.

// Words [K0, K1) of sw, at p (aligned to the vector).
template <int K0, int K1>
__host__ __device__ __forceinline__ void store_words(char* p, const uint32_t* sw) {
    if constexpr (K0 < K1) {
        constexpr int n = (K0 % 4 == 0 && K1 - K0 >= 4) ? 4 : (K0 % 2 == 0 && K1 - K0 >= 2) ? 2 : 1;
        if constexpr (n == 4)
            *reinterpret_cast<uint4*>(p + 4 * K0) = make_uint4(sw[K0], sw[K0 + 1], sw[K0 + 2], sw[K0 + 3]);
        else if constexpr (n == 2)
            *reinterpret_cast<uint2*>(p + 4 * K0) = make_uint2(sw[K0], sw[K0 + 1]);
        else
            *reinterpret_cast<uint32_t*>(p + 4 * K0) = sw[K0];
        store_words<K0 + n, K1>(p, sw);
    }
}

// Elements [LO, HI) of the vector whose words are sw.
template <typename T, int LO, int HI>
__host__ __device__ __forceinline__ void store_span(char* p, const uint32_t* sw) {
    if constexpr (sizeof(T) == 2) {
        if constexpr (LO & 1)  // element LO: the high half of word LO / 2
            *reinterpret_cast<unsigned short*>(p + 2 * LO) = static_cast<unsigned short>(sw[LO >> 1] >> 16);
        store_words<(LO + 1) / 2, HI / 2>(p, sw);
        if constexpr (HI & 1)  // element HI - 1: the low half of word HI / 2
            *reinterpret_cast<unsigned short*>(p + 2 * (HI - 1)) = static_cast<unsigned short>(sw[HI >> 1] & 0xffffu);
    } else {
        store_words<LO, HI>(p, sw);
    }
}

// The range by value: HI runs over VE, then the odd ends above LO.
template <typename T, int VE, int LO, int HI>
__host__ __device__ __forceinline__ void store_span_hi(char* p, const uint32_t* sw, int hi) {
    if constexpr (HI <= VE) {
        if (hi == HI) {
            store_span<T, LO, HI>(p, sw);
            return;
        }
        constexpr int first_odd = (LO & 1) ? LO + 2 : 1;
        constexpr int next = HI == VE ? first_odd : HI + 2;
        if constexpr (next < VE) store_span_hi<T, VE, LO, next>(p, sw, hi);
    }
}

// LO is 0 or 1.
template <typename T, int VE>
__host__ __device__ __forceinline__ void store_span_lo(char* p, const uint32_t* sw, int lo, int hi) {
    if (lo == 0) store_span_hi<T, VE, 0, VE>(p, sw, hi);
    else store_span_hi<T, VE, 1, VE>(p, sw, hi);
}

template <typename T, int V, int U, int DIR, bool RHEAD>
__global__ void __launch_bounds__(kThreads, kOddBlocksPerSm) rope_partial_odd_kernel(const KernelArgs a) {
    using P = Pack<T>;
    constexpr int W = V / 4;             // words per vector
    constexpr int WPP = P::kWordsPerPair;
    constexpr int PV = W / WPP;          // pair slots per lane
    constexpr int VE = 2 * PV;           // elements per vector
    static_assert(PV >= 1, "a vector holds at least one pair slot");
    const int npairs = a.pairs;          // pairs per row slice
    const bool wide = a.odd_wide != 0;
    const uint32_t C = a.divC.d;         // lanes per row
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t stride = uint64_t(gridDim.x) * kThreads;

    enter_after_predecessor();
    // Whole warps run the loop together, so every shuffle takes all 32
    // lanes; a lane past the end of the work ("dead") reads and writes
    // nothing.  tasks is a multiple of C, so a live lane's next lane in the
    // same row is live too (or in the next warp).
    for (uint64_t base = uint64_t(blockIdx.x) * kThreads + (threadIdx.x & ~31u); base < a.tasks;
         base += stride) {
        const bool live = base + lane < a.tasks;
        const uint32_t t = uint32_t(live ? base + lane : base);
        uint32_t rest, j, tok, hg, b, s;
        a.divC.divmod(t, rest, j);
        a.divH.divmod(rest, tok, hg);
        a.divS.divmod(tok, b, s);

        const int w0 = int(j) * PV;                   // slice pair of lane pair 0
        const int m_hi = npairs - w0 < PV ? npairs - w0 : PV;  // lane pairs [0, m_hi) are in the slice
        // element 0 is in the slice and its pair's first element is in the
        // previous lane of this warp (which sends the result up)
        const bool prev_here = j > 0 && lane != 0u;
        const bool ends_next = m_hi == PV;            // pair PV-1 ends in the next vector
        // ... and this lane stores that element: no next lane in the row, or
        // the next lane is in another warp
        const bool store_next = ends_next && (j + 1 == C || lane == 31u);
        // the elements of its vector the lane stores: all of them, or (a row's
        // edge lanes) [lo_e, hi_e)
        const int lo_e = prev_here ? 0 : 1;
        const int hi_e = 2 * m_hi + 1 < VE ? 2 * m_hi + 1 : VE;
        const bool full = lo_e == 0 && hi_e == VE;
        const int n0 = int(hg) * U;
        char* v0p = a.x + int64_t(tok) * a.tok_bytes + int64_t(n0) * a.row_bytes + int64_t(j) * V;
        const char* c_row = a.r1 + int64_t(b) * a.r1_b + int64_t(s) * a.r1_s;
        const char* s_row = a.r2 + int64_t(b) * a.r2_b + int64_t(s) * a.r2_s;
        if constexpr (RHEAD) {
            c_row += int64_t(n0) * a.r1_n;
            s_row += int64_t(n0) * a.r2_n;
        }

        // loads (dead lanes and heads past N read nothing and hold zeros)
        Words<W> xv[U];
        uint32_t xn[U];  // the next vector's first word, where this lane stores into it
#pragma unroll
        for (int i = 0; i < U; ++i) {
            xv[i] = Words<W>{};
            xn[i] = 0u;
            if (live && (i == 0 || n0 + i < a.N)) {
                char* p = v0p + int64_t(i) * a.row_bytes;
                xv[i] = ld_vec<W>(p);
                if (store_next) xn[i] = ld_vec<1>(p + V).w[0];
            }
        }
        Words<W> cv{}, sv{};
        if constexpr (!RHEAD) {
            if (live) {
                cv = load_lane_r<T, V>(c_row, w0, m_hi, wide);
                sv = load_lane_r<T, V>(s_row, w0, m_hi, wide);
            }
        }

#pragma unroll
        for (int i = 0; i < U; ++i) {
            const bool head = live && (i == 0 || n0 + i < a.N);
            const uint32_t down = __shfl_down_sync(0xffffffffu, xv[i].w[0], 1);
            uint32_t xw[W + 1];
#pragma unroll
            for (int k = 0; k < W; ++k) xw[k] = xv[i].w[k];
            xw[W] = store_next ? xn[i] : down;
            if constexpr (RHEAD) {
                if (head) {
                    cv = load_lane_r<T, V>(c_row + int64_t(i) * a.r1_n, w0, m_hi, wide);
                    sv = load_lane_r<T, V>(s_row + int64_t(i) * a.r2_n, w0, m_hi, wide);
                }
            }

            // the lane's pairs: f0[m], f1[m] are pair m's first and second
            // results in fp32
            float f0[PV], f1[PV];
#pragma unroll
            for (int m = 0; m < PV; ++m) {
                float x0, x1, c0, c1, s0, s1;
                odd_pair_x<T, W>(xw, m, x0, x1);
                P::get(&cv.w[m * WPP], c0, c1);
                P::get(&sv.w[m * WPP], s0, s1);
                rotate_pair<DIR>(x0, x1, c0, c1, s0, s1, f0[m], f1[m]);
            }
            // element 0: the previous lane's last second result
            const float prev = __uint_as_float(__shfl_up_sync(0xffffffffu, __float_as_uint(f1[PV - 1]), 1));

            // the vector as stored: word k holds elements 2k and 2k + 1, the
            // second result of pair k - 1 and the first of pair k (16-bit),
            // or element k (fp32)
            uint32_t sw[W];
            if constexpr (sizeof(T) == 2) {
                P::put(&sw[0], prev, f0[0]);
#pragma unroll
                for (int k = 1; k < W; ++k) P::put(&sw[k], f1[k - 1], f0[k]);
            } else {
                sw[0] = __float_as_uint(prev);
#pragma unroll
                for (int m = 0; m < PV; ++m) {
                    sw[2 * m + 1] = __float_as_uint(f0[m]);
                    if (2 * m + 2 < W) sw[2 * m + 2] = __float_as_uint(f1[m]);
                }
            }
            if (head) {
                char* p = v0p + int64_t(i) * a.row_bytes;
                if (full) {
                    Words<W> o;
#pragma unroll
                    for (int k = 0; k < W; ++k) o.w[k] = sw[k];
                    st_vec<W>(p, o);
                } else {
                    store_span_lo<T, VE>(p, sw, lo_e, hi_e);
                }
                // the last pair's second result opens the next vector
                if (store_next) {
                    if constexpr (sizeof(T) == 2)
                        *reinterpret_cast<unsigned short*>(p + V) = static_cast<unsigned short>(Elem<T>::put(f1[PV - 1]));
                    else
                        *reinterpret_cast<uint32_t*>(p + V) = __float_as_uint(f1[PV - 1]);
                }
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
// 1/(2*pi) minus inv_two_pi(), rounded to fp32 (1/(2*pi) =
// 0.159154943091895335768883763372514362...)
__device__ __forceinline__ float inv_two_pi_lo() { return __uint_as_float(0x31dc9c88u); } // 6.4206382e-09

// cos and sin of theta = p * omega, omega = hi + lo.  theta is carried as
// th + tl (th = p*hi rounded; tl = the exact residual of that product plus
// p*lo), accurate to about 2^-44 relative for |p| < 2^24 (p is then exact in
// fp32).  Reduction by 2*pi follows Cody and Waite ("Software Manual for the
// Elementary Functions", 1980) with the three-part constant above.  The
// multiple n is the integer nearest theta / (2*pi), taken from the quotient
// as a two-part sum (the rounded product th * (1/2pi), its exact residual,
// the constant's tail and tl's share), so that the reduced angle stays in
// [-pi, pi] up to rounding: a plain rintf(th * (1/2pi)) can be one off when
// |theta| is near 2^24, leaving |r| up to about 4.9, where the hardware
// sine's error bound does not hold.  Then r = ((th - n*A) - n*B) - n*C + tl,
// where the first step is exact (Sterbenz when |th| < 4, otherwise both
// terms are multiples of the first part's ulp and the difference has at most
// 23 bits).  The other three steps round once each, so |r - (theta - 2*pi*n)|
// <= 3 * 2^-23 (an fp32 emulation of these steps over 2^24-wide position
// ranges and bases 2 to 10^6 measured at most 2.6e-7).  On [-pi, pi] the
// hardware __sincosf has an absolute error of at most 2^-21.41 (CUDA's
// documented bound), so the cos/sin used are within about 7e-7 of the exact
// values (the GPU test of this bound asserts 8e-7), at a few instructions
// per angle.
__device__ __forceinline__ void angle_cos_sin(float p, float w_hi, float w_lo, float& c, float& s) {
    const float th = __fmul_rn(p, w_hi);
    const float tl = __fmaf_rn(p, w_lo, __fmaf_rn(p, w_hi, -th));
    const float q_hi = __fmul_rn(th, inv_two_pi());
    float q_lo = __fmaf_rn(th, inv_two_pi(), -q_hi);
    q_lo = __fmaf_rn(th, inv_two_pi_lo(), q_lo);
    q_lo = __fmaf_rn(tl, inv_two_pi(), q_lo);
    float n = rintf(q_hi);
    const float f = __fadd_rn(__fsub_rn(q_hi, n), q_lo);  // theta / (2*pi) - n
    n = f > 0.5f ? n + 1.0f : (f < -0.5f ? n - 1.0f : n);
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
        if (f)
            return p.r_head ? reinterpret_cast<const void*>(&rope_partial_odd_kernel<T, VEC, U, kFwd, true>)
                            : reinterpret_cast<const void*>(&rope_partial_odd_kernel<T, VEC, U, kFwd, false>);
        return p.r_head ? reinterpret_cast<const void*>(&rope_partial_odd_kernel<T, VEC, U, kBwd, true>)
                        : reinterpret_cast<const void*>(&rope_partial_odd_kernel<T, VEC, U, kBwd, false>);
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
        switch (p.vec) {
            case 16: return pick_heads<T, 16, false, kOdd>(p);
            case 8: return pick_heads<T, 8, false, kOdd>(p);
            default: return nullptr;
        }
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

/*
 * rope_partial.h -- C ABI of the GB300 in-place partial interleaved rotary
 * position embedding (inplace_partial_rotary_mul, forward and backward).
 *
 * Operation ("CANN ops-transformer inplace_partial_rotary_mul",
 * mhpn.cn/news/2302710, section 功能与计算公式): x is a contiguous tensor of
 * shape (B, S, N, D) ("BSND": batch, sequence, heads, head dim).  Only the
 * lanes [start, end) of its last axis change.  With L = end - start and the
 * lanes counted from start, each pair (2i, 2i+1) of the slice becomes
 *
 *     y[2i]   = x[2i]   * c[2i]   - x[2i+1] * s[2i]
 *     y[2i+1] = x[2i+1] * c[2i+1] + x[2i]   * s[2i+1]
 *
 * i.e. x_out = x_slice * cos + x_rotate * sin, where x_rotate swaps each pair
 * (the XOR-1 gather) and negates its even lanes; c comes from r1 (cos) and
 * s from r2 (sin).  The result is written back into x.
 *
 * The backward applies the transposed rotation to the incoming gradient g,
 * in place (same page, section 自动微分说明; the inverse rotation of
 * "ANE实战 RoPE位置编码在MIL中的纯ANE实现", section 反向传播):
 *
 *     dx[2i]   = g[2i]   * c[2i]   + g[2i+1] * s[2i+1]
 *     dx[2i+1] = g[2i+1] * c[2i+1] - g[2i]   * s[2i]
 *
 * Arithmetic: every input is widened to fp32; each product is one fp32
 * rounding and the sum is one fp32 rounding (no fused multiply-add); the
 * result is rounded once to the storage type, round-to-nearest-even (the
 * CAST_RINT write-back of the page's tiling section).  Results are
 * deterministic: no atomics, no reductions.
 *
 * Memory: every pointer is a device pointer (or managed memory) on the
 * current CUDA device; the *_host entry points below take host buffers.
 * The caller owns every buffer; the library allocates nothing and needs no
 * workspace.  Calls are asynchronous on `stream` and never synchronise.
 *
 * Error behaviour: arguments are validated on the host before anything is
 * launched; an invalid call changes nothing and returns an error status.
 * A call whose work is empty (end == start, or any of B, S, N, D is 0)
 * returns ROPE_OK without a launch and then accepts null data pointers
 * (the page's no-op rule for an empty slice or empty tensor).
 * rope_last_error_message() describes the most recent failure on the
 * calling thread.
 */
#ifndef ROPE_PARTIAL_H
#define ROPE_PARTIAL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t (a CUDA runtime stream handle); 0 is the
   legacy default stream. */
typedef struct CUstream_st* rope_stream_t;

/* Storage types of x, r1 and r2 (the three the page registers). */
typedef enum {
    ROPE_BF16 = 0,
    ROPE_FP16 = 1,
    ROPE_FP32 = 2
} rope_dtype_t;

/* Rotary modes.  Interleave is the page's mode and numbering (the ACLNN
   interface passes rotary_mode = 1 for interleave): lanes (2i, 2i+1) of the
   slice form a pair.  Half-split pairs lane i with lane i + L/2, reading the
   page's x_rotate = cat(-x2, x1) with x1, x2 the two halves of the slice,
   which is rotate_half of "ANE实战 RoPE位置编码在MIL中的纯ANE实现" (section
   先搞懂RoPE: swap the two halves and negate the front half). */
typedef enum {
    ROPE_MODE_INTERLEAVE = 1,
    ROPE_MODE_HALF = 2
} rope_mode_t;

/* Status codes (split after the aclnn null-pointer / invalid-parameter /
   internal-error convention). */
typedef enum {
    ROPE_OK = 0,
    ROPE_ERR_NULLPTR = 1, /* a required pointer is null                       */
    ROPE_ERR_INVALID = 2, /* dtype, sizes, slice, broadcast, stride or align   */
    ROPE_ERR_CUDA = 3     /* the launch or a device query failed               */
} rope_status_t;

/*
 * rope_partial_inplace_fwd -- rotate x[..., start:end) in place.
 *
 *   x          device pointer to a contiguous (B, S, N, D) tensor of `dtype`,
 *              read and written.  Aligned to its element size.
 *   r1, r2     device pointers to cos and sin: 4-D tensors of `dtype` with
 *              shape rX_shape[0..3] and ELEMENT strides rX_stride[0..3].
 *              Each of rX_shape[0..2] is 1 (broadcast; its stride is then
 *              ignored) or equal to B, S, N respectively; rX_shape[3] == L.
 *              rX_stride[3] must be 1 and the other strides >= 0.  r1 and r2
 *              are only read and must not overlap x: a call whose x shares a
 *              byte with r1 or r2 (from its first element to the end of its
 *              farthest row) returns ROPE_ERR_INVALID.
 *   B, S, N, D sizes of x, each >= 0; D even and D <= 1024.
 *   start, end 0 <= start <= end <= D and L = end - start even.  start may be
 *              odd: pairs are counted from start.
 *   stream     the CUDA stream to launch on.
 *
 * Returns ROPE_OK after the launch was queued (or for an empty call),
 * ROPE_ERR_NULLPTR for a null x / r1 / r2 / shape / stride pointer when
 * there is work, ROPE_ERR_INVALID when a rule above is broken, and
 * ROPE_ERR_CUDA when the launch fails.
 */
rope_status_t rope_partial_inplace_fwd(void* x, const void* r1, const void* r2,
                                       rope_dtype_t dtype, int64_t B, int64_t S,
                                       int64_t N, int64_t D,
                                       const int64_t r1_shape[4], const int64_t r1_stride[4],
                                       const int64_t r2_shape[4], const int64_t r2_stride[4],
                                       int64_t start, int64_t end, rope_stream_t stream);

/*
 * rope_partial_inplace_bwd -- overwrite grad[..., start:end) with the
 * gradient with respect to x of the forward above (the transposed rotation).
 * Arguments, layout, ownership and errors are those of the forward, with
 * `grad` (the incoming gradient, shape (B, S, N, D)) in place of x.  r1 and
 * r2 get no gradient.
 */
rope_status_t rope_partial_inplace_bwd(void* grad, const void* r1, const void* r2,
                                       rope_dtype_t dtype, int64_t B, int64_t S,
                                       int64_t N, int64_t D,
                                       const int64_t r1_shape[4], const int64_t r1_stride[4],
                                       const int64_t r2_shape[4], const int64_t r2_stride[4],
                                       int64_t start, int64_t end, rope_stream_t stream);

/*
 * rope_partial_inplace_fwd_mode / rope_partial_inplace_bwd_mode -- the
 * forward and backward above with an explicit rotary mode.  With
 * ROPE_MODE_INTERLEAVE they are rope_partial_inplace_fwd / _bwd.  With
 * ROPE_MODE_HALF, for j in [0, L/2) and m = j, n = j + L/2 (slice-relative):
 *     y[m] = x[m] * c[m] - x[n] * s[m]        dx[m] = g[m] * c[m] + g[n] * s[n]
 *     y[n] = x[n] * c[n] + x[m] * s[n]        dx[n] = g[n] * c[n] - g[m] * s[m]
 * with the same rounding, validation and errors (an unknown mode returns
 * ROPE_ERR_INVALID).
 */
rope_status_t rope_partial_inplace_fwd_mode(void* x, const void* r1, const void* r2,
                                            rope_dtype_t dtype, int64_t B, int64_t S,
                                            int64_t N, int64_t D,
                                            const int64_t r1_shape[4], const int64_t r1_stride[4],
                                            const int64_t r2_shape[4], const int64_t r2_stride[4],
                                            int64_t start, int64_t end, rope_mode_t mode,
                                            rope_stream_t stream);

rope_status_t rope_partial_inplace_bwd_mode(void* grad, const void* r1, const void* r2,
                                            rope_dtype_t dtype, int64_t B, int64_t S,
                                            int64_t N, int64_t D,
                                            const int64_t r1_shape[4], const int64_t r1_stride[4],
                                            const int64_t r2_shape[4], const int64_t r2_stride[4],
                                            int64_t start, int64_t end, rope_mode_t mode,
                                            rope_stream_t stream);

/*
 * rope_partial_inplace_fwd_pos / rope_partial_inplace_bwd_pos -- the same
 * operations with cos and sin computed in the kernel from positions instead
 * of read from r1 / r2.  The angle of pair k in [0, L/2) at position p is
 * theta_k = p / base^(2k/L) (the RoPE definition and table recipe of
 * "ANE实战 RoPE位置编码在MIL中的纯ANE实现", sections 先搞懂RoPE and 第一步,
 * base 10000 there); both lanes of the pair use cos(theta_k) and
 * sin(theta_k), i.e. the pair-duplicated table (interleave) or the
 * half-duplicated one (half), without the table's bytes.
 *
 *   positions  device pointer to int32 positions, one per (batch, seq), of
 *              shape pos_shape[0..1] (each 1 or B, S respectively) with
 *              ELEMENT strides pos_stride[0..1]; read only.  The error
 *              bound below holds for |p| < 2^24, where p is exact in fp32;
 *              a larger position is rounded to fp32 before use, and the
 *              reduction by 2*pi then loses that bound (the call still
 *              runs; nothing on the device checks the range).
 *   base       > 0 and finite (10000 in the usual recipe).
 *   mode       ROPE_MODE_INTERLEAVE or ROPE_MODE_HALF.
 *   other      as for rope_partial_inplace_fwd (x / grad, sizes, slice,
 *              stream, asynchrony, the empty-call rule, status codes).
 *
 * Arithmetic: omega_k = base^(-2k/L) is computed on the host in double and
 * passed as two fp32 parts; theta is formed and reduced by 2*pi in fp32
 * arithmetic that keeps its error within 3 * 2^-23 (see the kernel), and the
 * hardware sine/cosine on the reduced angle gives cos and sin to within
 * 8e-7 of the exact values (for |p| < 2^24).  They stay in fp32 (they are
 * not rounded to x's type); the rotation then rounds as above.  Results are therefore within that bound
 * of the same operation with an fp32 table of correctly rounded cos/sin,
 * not bit-identical to it.
 */
rope_status_t rope_partial_inplace_fwd_pos(void* x, const int32_t* positions, rope_dtype_t dtype,
                                           int64_t B, int64_t S, int64_t N, int64_t D,
                                           const int64_t pos_shape[2], const int64_t pos_stride[2],
                                           double base, int64_t start, int64_t end,
                                           rope_mode_t mode, rope_stream_t stream);

rope_status_t rope_partial_inplace_bwd_pos(void* grad, const int32_t* positions,
                                           rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                           int64_t D, const int64_t pos_shape[2],
                                           const int64_t pos_stride[2], double base,
                                           int64_t start, int64_t end, rope_mode_t mode,
                                           rope_stream_t stream);

/*
 * rope_partial_inplace_fwd_qk / rope_partial_inplace_bwd_qk -- one launch
 * that rotates a query slice and a key slice with the same cos/sin rows: the
 * RoPE stage of MLA preprocessing, which applies the rotation to
 * Q[..., :qRopeDim] and K[..., :kRopeDim] with cos/sin of one row per token
 * ("ascend-transformer-boost MlaPreprocessOperation", m.xxqk.cn/news/384935,
 * sections 3 and 4).  The result equals rope_partial_inplace_fwd on q
 * followed by rope_partial_inplace_fwd on k (backward: _bwd on dq and dk), in
 * one launch that reads each cos/sin row once for both.
 *
 *   q, k       device pointers to contiguous (B, S, Nq, Dq) and (B, S, Nk, Dk)
 *              tensors of `dtype` (the key may have its own head count and
 *              head dim); both are read and written, so they must not share a
 *              byte (ROPE_ERR_INVALID), nor may either share one with r1/r2.
 *   q_start/q_end, k_start/k_end
 *              the two slices; same rules as `start`/`end` above, and the same
 *              length L = q_end - q_start = k_end - k_start.
 *   r1, r2     cos and sin as above with rX_shape[2] == 1 (one row per
 *              (batch, position), shared by every query and key head).
 *
 * Validation, ownership, asynchrony and status codes are those of
 * rope_partial_inplace_fwd; a tensor whose work is empty is skipped.
 */
rope_status_t rope_partial_inplace_fwd_qk(void* q, void* k, const void* r1, const void* r2,
                                          rope_dtype_t dtype, int64_t B, int64_t S,
                                          int64_t Nq, int64_t Dq, int64_t q_start, int64_t q_end,
                                          int64_t Nk, int64_t Dk, int64_t k_start, int64_t k_end,
                                          const int64_t r1_shape[4], const int64_t r1_stride[4],
                                          const int64_t r2_shape[4], const int64_t r2_stride[4],
                                          rope_stream_t stream);

rope_status_t rope_partial_inplace_bwd_qk(void* dq, void* dk, const void* r1, const void* r2,
                                          rope_dtype_t dtype, int64_t B, int64_t S,
                                          int64_t Nq, int64_t Dq, int64_t q_start, int64_t q_end,
                                          int64_t Nk, int64_t Dk, int64_t k_start, int64_t k_end,
                                          const int64_t r1_shape[4], const int64_t r1_stride[4],
                                          const int64_t r2_shape[4], const int64_t r2_stride[4],
                                          rope_stream_t stream);

/*
 * rope_partial_inplace_fwd_host / rope_partial_inplace_bwd_host -- the same
 * operations on buffers in HOST memory, which the kernel reads and writes in
 * place across the host link (zero copy: no device buffer, no staging copy).
 * On Grace-Blackwell the GPU reaches host memory coherently over NVLink-C2C,
 * so only the slice bytes and the cos/sin rows cross the link, instead of
 * whole tensors copied both ways.
 *
 * Arguments and layout are those of rope_partial_inplace_fwd / _bwd.  x (or
 * grad), r1 and r2 must be memory the current device can access: page-locked
 * host memory (cudaHostAlloc / cudaMallocHost, or registered with
 * cudaHostRegister), managed memory, device memory, or -- on a device that
 * reports cudaDevAttrPageableMemoryAccess -- any host memory.  The first and
 * last byte of each buffer are checked with cudaPointerGetAttributes before
 * anything is launched; a buffer the device cannot reach returns
 * ROPE_ERR_INVALID.  The call is asynchronous: synchronise `stream` before
 * the host reads x.
 */
rope_status_t rope_partial_inplace_fwd_host(void* x, const void* r1, const void* r2,
                                            rope_dtype_t dtype, int64_t B, int64_t S,
                                            int64_t N, int64_t D,
                                            const int64_t r1_shape[4], const int64_t r1_stride[4],
                                            const int64_t r2_shape[4], const int64_t r2_stride[4],
                                            int64_t start, int64_t end, rope_stream_t stream);

rope_status_t rope_partial_inplace_bwd_host(void* grad, const void* r1, const void* r2,
                                            rope_dtype_t dtype, int64_t B, int64_t S,
                                            int64_t N, int64_t D,
                                            const int64_t r1_shape[4], const int64_t r1_stride[4],
                                            const int64_t r2_shape[4], const int64_t r2_stride[4],
                                            int64_t start, int64_t end, rope_stream_t stream);

/*
 * Data-parallel split of the token grid (multi-GPU: one process per GPU,
 * no collective).  Every row (b, s, n) of the operation needs only itself
 * and its own cos/sin row, so the tokens t = b * S + s of one workload can
 * be split across ranks with nothing exchanged: each rank rotates its own
 * tokens' rows with its own cos/sin rows.  This follows the token-range
 * convention of "CANN ops-transformer aclnnMoeTokenUnpermuteWithEpGrad"
 * (lshu.cn/news/80967, section 一: under expert-parallel splitting each
 * device handles only the tokens in [range[0], range[1])).
 *
 * rope_partial_token_shard gives rank `rank` of `world` the tokens
 * [*t0, *t1) of a (B, S) grid: contiguous in b * S + s order, the first
 * (B * S) % world ranks one token more than the others, the ranks in order
 * tiling [0, B * S) exactly once.  It splits that range into *nruns <= 3
 * runs, in order, each a contiguous block of a BSND tensor that one call of
 * this library can rotate: the end of a batch entered mid-way, whole
 * batches, the start of a batch (a range inside one batch is one run).
 * Run k covers batches [b0, b0 + nb) x positions [s0, s0 + ns), and either
 * nb == 1 or (s0 == 0 and ns == S).  For that call, x starts at token
 * (b0, s0) (byte offset (b0 * S + s0) * N * D * e of the full tensor, or of
 * the rank's own buffer of its tokens at ((b0 * S + s0) - t0) * N * D * e),
 * the sizes are (nb, ns, N, D), and cos/sin start at their (b0, s0) row
 * along each dim they do not broadcast, shapes (nb or 1, ns or 1, Nr, L),
 * strides unchanged.
 *
 * Host only: no CUDA call.  B, S >= 0, 0 <= rank < world.  An empty grid
 * or an empty share gives *nruns == 0 and *t0 == *t1.  Returns
 * ROPE_ERR_NULLPTR for a null output pointer, ROPE_ERR_INVALID for
 * negative sizes, a rank outside [0, world) or a B * S that overflows.
 */
typedef struct {
    int64_t b0; /* first batch of the run                                    */
    int64_t s0; /* first position (sequence index) in each of its batches    */
    int64_t nb; /* batches: 1, or several whole batches                      */
    int64_t ns; /* positions per batch of the run (S whenever nb > 1)         */
} rope_token_run_t;

rope_status_t rope_partial_token_shard(int64_t B, int64_t S, int32_t rank, int32_t world,
                                       int64_t* t0, int64_t* t1, rope_token_run_t runs[3],
                                       int32_t* nruns);

/* A static, human-readable name of a status code. */
const char* rope_status_str(rope_status_t status);

/* A description of the most recent non-OK status returned on the calling
   thread ("" if none).  The string stays valid until the thread's next call. */
const char* rope_last_error_message(void);

/*
 * Launch plan, for inspection and tests.  rope_partial_plan validates the
 * same arguments as the forward (data pointers are used only for their
 * alignment and may be any value with the alignment they will have) and
 * reports the kernel the call would launch.  sm_count > 0 sizes the grid
 * for that many SMs without touching the GPU; sm_count == 0 asks the current
 * device.  No kernel is launched.
 */
typedef struct {
    int32_t path;             /* 0: no launch (empty), 1: vector kernel, 2: scalar-pair kernel, */
                              /* 3: half-split vector kernel whose row of accesses fits one     */
                              /* warp (the partner access comes from another lane), 4:          */
                              /* interleave with an odd start at element 1 of an aligned        */
                              /* vector, a lane per 16- or 8-byte vector of x                   */
    int32_t vec_bytes;        /* bytes per global access of x (16, 8 or 4; on the scalar path  */
                              /* a pair (interleave) or an element (half-split))                */
    int32_t heads_per_thread; /* heads one thread walks with its cos/sin kept in registers     */
    int32_t threads_per_block;
    int64_t blocks;           /* grid size                                                    */
    int64_t tasks;            /* (token, head group, chunk) work items                        */
    int32_t chunks_per_row;   /* accesses covering one row's slice                            */
    int32_t r_per_head;       /* 1 when cos/sin differ between heads (reloaded per head)       */
    int64_t launches;         /* kernel launches: calls whose work index would pass 2^31 are   */
                              /* split into launches over whole batches or runs of tokens       */
} rope_plan_t;

rope_status_t rope_partial_plan(const void* x, const void* r1, const void* r2,
                                rope_dtype_t dtype, int64_t B, int64_t S, int64_t N, int64_t D,
                                const int64_t r1_shape[4], const int64_t r1_stride[4],
                                const int64_t r2_shape[4], const int64_t r2_stride[4],
                                int64_t start, int64_t end, int32_t sm_count,
                                rope_plan_t* plan);

/* The plan of rope_partial_inplace_fwd_mode (rope_partial_plan is this with
   ROPE_MODE_INTERLEAVE). */
rope_status_t rope_partial_plan_mode(const void* x, const void* r1, const void* r2,
                                     rope_dtype_t dtype, int64_t B, int64_t S, int64_t N,
                                     int64_t D, const int64_t r1_shape[4],
                                     const int64_t r1_stride[4], const int64_t r2_shape[4],
                                     const int64_t r2_stride[4], int64_t start, int64_t end,
                                     rope_mode_t mode, int32_t sm_count, rope_plan_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* ROPE_PARTIAL_H */

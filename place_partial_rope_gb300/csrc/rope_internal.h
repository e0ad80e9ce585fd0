// rope_internal.h -- what the host planner hands to the launcher.
// Not part of the public ABI (that is include/rope_partial.h).
#pragma once
#include <stdint.h>

#include "fast_div.h"
#include "rope_partial.h"

namespace rope {

constexpr int kThreads = 256;            // threads per block
constexpr int kBlocksPerSmCap = 8;       // 2048 resident threads per SM / 256
// The odd-start kernel's launch bound: at least 4 resident blocks per SM
// (64 registers a thread).  Back to back on GB300 this ran the GQA shape's
// [1, 65) forward in 58.0 us against 64.6 us without it (68 registers, 3
// blocks per SM) and 81 us with 5 blocks (spills).
constexpr int kOddBlocksPerSm = 4;
constexpr uint32_t kMaxPieceTasks = 1u << 31;  // flat work index of one launch
constexpr int kMaxPairs = 512;           // L / 2 for the largest slice (D <= 1024)

// Rotation frequencies of the positions call, omega_k = base^(-2k/L), each
// as an fp32 pair hi + lo (hi = omega rounded to fp32, lo = the remainder
// rounded to fp32), passed by value as the kernel's second parameter.
struct FreqTable {
    float hi[kMaxPairs];
    float lo[kMaxPairs];
};

enum Direction : int { kFwd = 0, kBwd = 1 };
enum Path : int { kNone = 0, kVector = 1, kScalarPair = 2, kOddPair = 4 };
enum Mode : int { kInterleave = 1, kHalf = 2 };  // the ACLNN numbering: interleave = 1

// What one launch covers: a contiguous range of tokens ("a piece").  The
// kernel turns its flat work index into (token, head group, chunk) with
// three fast divisions, then into byte offsets from the piece's bases.
struct KernelArgs {
    char* x;                   // row 0 of the piece's first token, plus start * e
                               // (odd-start kernel: plus (start - 1) * e, the
                               // vector that holds element start)
    const char* r1;            // cos of the piece's first (batch, seq) position
    const char* r2;            // sin of the same
    int64_t tok_bytes;         // bytes between consecutive tokens of x (N * D * e)
    int64_t row_bytes;         // bytes between consecutive heads of x (D * e)
    int64_t r1_b, r1_s, r1_n;  // byte strides of r1 for batch, seq, head (0: broadcast)
    int64_t r2_b, r2_s, r2_n;
    char* x2;                  // fused query + key call: row 0 of the second tensor's
                               // piece, plus its slice offset (nullptr otherwise)
    int64_t tok_bytes2;        // token pitch of the second tensor
    int64_t row_bytes2;        // head pitch of the second tensor
    int64_t half_off;          // half-split mode: bytes from lane j to lane j + L/2
    const int32_t* pos;        // positions call: position of the piece's first (b, s)
    int64_t pos_b, pos_s;      // element strides of the positions (0: broadcast)
    int32_t pairs;             // positions call: L / 2 entries of the FreqTable;
                               // odd-start kernel: pairs per row slice
    int32_t odd_wide;          // odd-start kernel: cos/sin rows aligned for one
                               // V-byte access per lane
    uint32_t tasks;            // work items of the piece: tokens * (H + H2) * C
    uint32_t tasks1;           // fused query + key call: the first tensor's items
                               // (tokens * H * C), which come before the second's
    int32_t N;                 // heads (first tensor's plus second tensor's)
    int32_t N1;                // heads of the first tensor
    int32_t H;                 // head groups of the first tensor = ceil(N1 / U);
                               // group hg holds heads hg*U .. hg*U + U - 1
    FastDiv divC;              // chunks per row
    FastDiv divH;              // head groups of the first tensor
    FastDiv divH2;             // head groups of the second tensor (ceil((N - N1) / U))
    FastDiv divS;              // tokens per batch inside the piece
};

// The kernel a validated call runs.
struct Plan {
    int dtype;      // rope_dtype_t
    int dir;        // Direction
    int path;       // Path
    int vec;        // bytes per access of x: 16, 8 or 4 (vector), 2 * e (scalar pair)
    int U;          // heads per thread (cos/sin reused from registers across them)
    int H;          // head groups (of the first tensor when there are two)
    int H2;         // head groups of the second tensor (0 when there is one)
    int C;          // chunks (accesses) per row slice
    bool r_head;    // cos/sin differ between heads: reloaded per head
    bool two;       // fused query + key call (rope_partial_qk_kernel)
    bool half;      // half-split mode (rope_partial_half_kernel)
    bool lanes;     // half-split with C accesses per row (a power of two in
                    // [2, 32]), the partner access in lane ^ C/2
                    // (rope_partial_half_lanes_kernel)
    bool full_grid; // one block per 256 work items instead of a resident,
                    // grid-striding grid
    bool pos;       // cos/sin computed from positions (rope_partial_pos_kernel)
    bool odd_wide;  // odd start (kOddPair): each lane's cos/sin is one aligned
                    // vec-byte access
};

// The kernel instance a plan runs, or nullptr if none was compiled for it
// (defined in the .cu; a table lookup, no CUDA call).
const void* kernel_lookup(const Plan& plan);

// Launch one piece on `stream` with `blocks` blocks (defined in the .cu);
// `freq` is the positions call's frequency table (nullptr otherwise).
rope_status_t launch_piece(const Plan& plan, const KernelArgs& args, const FreqTable* freq,
                           uint32_t blocks, rope_stream_t stream, const char** err);

// A device address for the buffer [p, p + bytes) when the current device
// can reach all of it (device, managed, page-locked host memory, or any host
// memory on a device with pageable-memory access); ROPE_ERR_INVALID when it
// cannot (defined in the .cu).
rope_status_t device_address(const void* p, int64_t bytes, const void** out, const char** err);

// The current device's SM count and the planned kernel's resident blocks
// per SM (defined in the .cu; the only device queries the library makes).
rope_status_t device_sm_count(int* sms, const char** err);
rope_status_t kernel_blocks_per_sm(const Plan& plan, int* blocks, const char** err);

}  // namespace rope

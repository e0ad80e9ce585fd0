// rope_kernels_bf16.cu -- the bf16 instances of rope_partial_kernel (one
// translation unit per storage type so the build compiles them in parallel).
#include "rope_kernels.cuh"

namespace rope {

const void* kernel_for_bf16(const Plan& p) { return pick_kernel<__nv_bfloat16>(p); }

}  // namespace rope

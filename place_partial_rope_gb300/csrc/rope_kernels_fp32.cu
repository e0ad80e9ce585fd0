// rope_kernels_fp32.cu -- the fp32 instances of rope_partial_kernel (one
// translation unit per storage type so the build compiles them in parallel).
#include "rope_kernels.cuh"

namespace rope {

const void* kernel_for_fp32(const Plan& p) { return pick_kernel<float>(p); }

}  // namespace rope

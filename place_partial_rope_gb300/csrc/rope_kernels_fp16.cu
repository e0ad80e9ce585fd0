// rope_kernels_fp16.cu -- the fp16 instances of rope_partial_kernel (one
// translation unit per storage type so the build compiles them in parallel).
#include "rope_kernels.cuh"

namespace rope {

const void* kernel_for_fp16(const Plan& p) { return pick_kernel<__half>(p); }

}  // namespace rope

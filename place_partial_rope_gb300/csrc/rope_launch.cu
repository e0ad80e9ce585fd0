// rope_launch.cu -- the library's only CUDA runtime calls: device and
// occupancy queries (cached) and the kernel launch on the caller's stream.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "rope_kernels.cuh"

namespace rope {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0 = not queried yet

std::mutex g_occ_mu;
std::unordered_map<const void*, int> g_occ[kMaxDevices];

const void* kernel_for(const Plan& p) {
    switch (p.dtype) {
        case ROPE_BF16: return kernel_for_bf16(p);
        case ROPE_FP16: return kernel_for_fp16(p);
        case ROPE_FP32: return kernel_for_fp32(p);
        default: return nullptr;
    }
}

rope_status_t cuda_fail(cudaError_t e, const char** err) {
    *err = cudaGetErrorString(e);
    (void)cudaGetLastError();  // leave no launch error behind for the caller
    return ROPE_ERR_CUDA;
}

// The address the current device uses to reach p (ROPE_ERR_INVALID when
// it cannot reach p).
rope_status_t resolve_one(const void* p, const void** out, const char** err) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) return cuda_fail(e, err);
    switch (a.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            *out = p;
            return ROPE_OK;
        case cudaMemoryTypeHost:
            if (a.devicePointer) {
                *out = a.devicePointer;
                return ROPE_OK;
            }
            *err = "page-locked host buffer is not mapped for the current device";
            return ROPE_ERR_INVALID;
        default: {  // unregistered (pageable) host memory
            int dev = 0, pageable = 0;
            e = cudaGetDevice(&dev);
            if (e != cudaSuccess) return cuda_fail(e, err);
            e = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
            if (e != cudaSuccess) return cuda_fail(e, err);
            if (pageable) {
                *out = p;
                return ROPE_OK;
            }
            *err = "pageable host buffer: this device cannot access it; use page-locked memory";
            return ROPE_ERR_INVALID;
        }
    }
}

}  // namespace

const void* kernel_lookup(const Plan& plan) { return kernel_for(plan); }

rope_status_t device_address(const void* p, int64_t bytes, const void** out, const char** err) {
    const void* first = nullptr;
    const void* last = nullptr;
    rope_status_t st = resolve_one(p, &first, err);
    if (st != ROPE_OK) return st;
    st = resolve_one(static_cast<const char*>(p) + (bytes > 0 ? bytes - 1 : 0), &last, err);
    if (st != ROPE_OK) return st;
    if (static_cast<const char*>(last) - static_cast<const char*>(first) != (bytes > 0 ? bytes - 1 : 0)) {
        *err = "buffer is not one contiguous device-accessible range";
        return ROPE_ERR_INVALID;
    }
    *out = first;
    return ROPE_OK;
}

rope_status_t device_sm_count(int* sms, const char** err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, err);
    if (dev >= 0 && dev < kMaxDevices) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) {
            *sms = cached;
            return ROPE_OK;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, err);
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    *sms = n;
    return ROPE_OK;
}

rope_status_t kernel_blocks_per_sm(const Plan& plan, int* blocks, const char** err) {
    const void* f = kernel_for(plan);
    if (!f) {
        *err = "internal error: no kernel instance for this plan";
        return ROPE_ERR_CUDA;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, err);
    const int slot = (dev >= 0 && dev < kMaxDevices) ? dev : 0;
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        auto it = g_occ[slot].find(f);
        if (it != g_occ[slot].end()) {
            *blocks = it->second;
            return ROPE_OK;
        }
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kThreads, 0);
    if (e != cudaSuccess) return cuda_fail(e, err);
    if (n > kBlocksPerSmCap) n = kBlocksPerSmCap;
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        g_occ[slot][f] = n;
    }
    *blocks = n;
    return ROPE_OK;
}

rope_status_t launch_piece(const Plan& plan, const KernelArgs& args, const FreqTable* freq,
                           uint32_t blocks, rope_stream_t stream, const char** err) {
    const void* f = kernel_for(plan);
    if (!f) {
        *err = "internal error: no kernel instance for this plan";
        return ROPE_ERR_CUDA;
    }
    if (blocks == 0) return ROPE_OK;
    KernelArgs a = args;
    // rope_partial_pos_kernel takes the frequency table as a second parameter
    void* params[] = {&a, const_cast<FreqTable*>(freq)};
    // programmatic dependent launch: the kernels wait (griddepcontrol.wait)
    // before their first global access, so the next launch may overlap the
    // tail of this one
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelExC(&cfg, f, params);
    if (e != cudaSuccess) return cuda_fail(e, err);
    return ROPE_OK;
}

}  // namespace rope

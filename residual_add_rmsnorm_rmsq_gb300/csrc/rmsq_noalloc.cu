// Allocation-free entry point for NVFP4 with a data-derived global scale.
//
// rmsq_fused_add_rmsnorm_nvfp4_dynamic needs a small device workspace (the
// batch amax word and one fp32 per row).  Some callers cannot provide one:
// code that gets no device allocator from its host (a plugin inside an
// engine that owns every byte of device memory through its own pool), or
// latency-critical code that must never call cudaMalloc because it can
// synchronise the device.  For them this entry point keeps the workspace in
// a fixed, file-scope device array and otherwise forwards to the regular
// entry point.
//
// The array is allocated with the module on every device that loads the
// library and stays until the process exits.  In host code its name only
// stands for the device symbol, so its device address is looked up once per
// device (cudaGetSymbolAddress, with that device current) and that address
// is what the kernels get.
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "rmsq.h"

namespace {

constexpr size_t kNoallocScratchBytes = 256 + 4 * static_cast<size_t>(RMSQ_NOALLOC_MAX_TOKENS);
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size is a multiple of 256");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 128;
std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mu;

// Device address of the scratch array on the current device (looked up on
// the first call per device).  Returns an rmsq_status.
int scratch_for_current_device(void** out) {
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
        cudaGetLastError();
        return RMSQ_ERR_NO_DEVICE;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RMSQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RMSQ_ERR_UNSUPPORTED_DEVICE;
    void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        p = g_scratch_ptr[dev].load(std::memory_order_acquire);
        if (!p) {
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) return RMSQ_ERR_CUDA;
            g_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return RMSQ_OK;
}

}  // namespace

extern "C" int rmsq_fused_add_rmsnorm_nvfp4_dynamic_noalloc(
    const void* x, const void* residual, const void* weight, float eps, void* out_q,
    void* out_block_scales, float* out_global_scale, void* residual_out, int64_t n_tokens,
    int64_t hidden, int dtype, void* stream, int variant) {
    if (n_tokens < 0) return RMSQ_ERR_INVALID_ARG;
    if (n_tokens > RMSQ_NOALLOC_MAX_TOKENS) return RMSQ_ERR_UNSUPPORTED_SHAPE;
    if (n_tokens == 0)
        return rmsq_fused_add_rmsnorm_nvfp4_dynamic(x, residual, weight, eps, out_q, out_block_scales,
                                                    out_global_scale, residual_out, nullptr, 0, 0, hidden,
                                                    dtype, stream, variant);
    void* scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != RMSQ_OK) return st;
    return rmsq_fused_add_rmsnorm_nvfp4_dynamic(x, residual, weight, eps, out_q, out_block_scales,
                                                out_global_scale, residual_out, scratch,
                                                kNoallocScratchBytes, n_tokens, hidden, dtype, stream,
                                                variant);
}

// Allocation-free entry point for NVFP4 with a data-derived global scale.
//
// rmsq_fused_add_rmsnorm_nvfp4_dynamic needs a small device workspace (the
// per-row inverse RMS and per-CTA partial maxima of the first pass).  Some callers cannot provide one:
// code that gets no device allocator from its host (a plugin inside an
// engine that owns every byte of device memory through its own pool), or
// latency-critical code that must never call cudaMalloc because it can
// synchronise the device.  For them this entry point keeps the workspace in
// a fixed, file-scope device array and otherwise forwards to the regular
// entry point.
//
// The array is allocated with the module on every device that loads the
// library and stays until the process exits (or until the device's primary
// context is reset, after which the module is loaded again, possibly at
// another address).  In host code its name only stands for the device
// symbol, so every call looks up its device address (cudaGetSymbolAddress,
// with the caller's device current; after the first call on a device this is
// a host-side table lookup) and that address is what the kernels get.  The
// first call on a device loads the module there if nothing else has.
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "rmsq.h"
#include "rmsq_abi.h"

namespace {

constexpr size_t kNoallocScratchBytes = 256 + 8 * static_cast<size_t>(RMSQ_NOALLOC_MAX_TOKENS);
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size is a multiple of 256");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch array in the current device's context.
// Returns an rmsq_status; a failed lookup is recorded for
// rmsq_last_cuda_error() and not left pending.
int scratch_for_current_device(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return rmsq_abi::fail_cuda(e);
    if (!p) return RMSQ_ERR_CUDA;
    *out = p;
    return RMSQ_OK;
}

}  // namespace

extern "C" int rmsq_fused_add_rmsnorm_nvfp4_dynamic_noalloc(
    const void* x, const void* residual, const void* weight, float eps, void* out_q,
    void* out_block_scales, float* out_global_scale, void* residual_out, int64_t n_tokens,
    int64_t hidden, int dtype, void* stream, int variant) {
    // Argument and device checks come before the symbol lookup, so that a bad
    // argument or another device gets the same status as from the entry point
    // with a workspace, which checks everything else before any launch.
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    if (variant != RMSQ_VARIANT_AUTO && variant != RMSQ_VARIANT_DIRECT && variant != RMSQ_VARIANT_PIPELINED)
        return RMSQ_ERR_INVALID_ARG;
    if (n_tokens < 0 || hidden <= 0 || !std::isfinite(eps) || eps < 0.0f) return RMSQ_ERR_INVALID_ARG;
    if (n_tokens > RMSQ_NOALLOC_MAX_TOKENS) return RMSQ_ERR_UNSUPPORTED_SHAPE;
    if (n_tokens == 0)
        return rmsq_fused_add_rmsnorm_nvfp4_dynamic(x, residual, weight, eps, out_q, out_block_scales,
                                                    out_global_scale, residual_out, nullptr, 0, 0, hidden,
                                                    dtype, stream, variant);
    int st = rmsq_abi::check_device();
    if (st != RMSQ_OK) return st;
    void* scratch = nullptr;
    st = scratch_for_current_device(&scratch);
    if (st != RMSQ_OK) return st;
    return rmsq_fused_add_rmsnorm_nvfp4_dynamic(x, residual, weight, eps, out_q, out_block_scales,
                                                out_global_scale, residual_out, scratch,
                                                kNoallocScratchBytes, n_tokens, hidden, dtype, stream,
                                                variant);
}

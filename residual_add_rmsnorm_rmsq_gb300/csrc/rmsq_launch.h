// Host-side launch interface shared by the C ABI and the per-dtype kernel units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rmsq {

struct LaunchArgs {
    const void* x;
    const void* res;        // nullptr: no residual add
    const void* w;
    void* res_out;
    void* q;
    void* scales;
    const float* scale_in;
    float eps;
    int mode;
    int n;
    int hidden;
};

// One launch of the row kernel for bf16 / fp16 activations.
cudaError_t launch_rows_bf16(const LaunchArgs& a, cudaStream_t stream);
cudaError_t launch_rows_fp16(const LaunchArgs& a, cudaStream_t stream);
cudaError_t launch_convert(int kind, const float* in, uint8_t* out, int64_t n, cudaStream_t stream);

}  // namespace rmsq

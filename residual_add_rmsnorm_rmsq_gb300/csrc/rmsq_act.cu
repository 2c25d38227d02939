// bf16 and fp16 instantiations of the SiLU+Mul + quantisation kernel.
#include "rmsq_dispatch.cuh"
#include "rmsq_act.cuh"

namespace rmsq {
cudaError_t launch_act_bf16(const LaunchArgs& a, cudaStream_t stream) { return launch_act<Bf16T>(a, true, stream); }
cudaError_t launch_act_fp16(const LaunchArgs& a, cudaStream_t stream) { return launch_act<Fp16T>(a, true, stream); }
cudaError_t launch_quant_bf16(const LaunchArgs& a, cudaStream_t stream) { return launch_act<Bf16T>(a, false, stream); }
cudaError_t launch_quant_fp16(const LaunchArgs& a, cudaStream_t stream) { return launch_act<Fp16T>(a, false, stream); }

// Same steps as the kernel, two elements per thread, for elementwise checks.
__global__ void debug_activation_kernel(int kind, const float* in, const float* in2, float* out, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 2;
    for (int64_t i = 2 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x); i < n; i += stride) {
        const bool two = i + 1 < n;
        const float2 x = make_float2(in[i], two ? in[i + 1] : 0.0f);
        float2 r;
        if (kind == 0) {
            r = exp_cw2(x);
        } else if (kind == 3) {
            r = exp_cw2_mid(x);
        } else {
            const float2 u = kind == 2 ? make_float2(in2[i], two ? in2[i + 1] : 0.0f) : make_float2(1.0f, 1.0f);
            r = kind == 2 ? silu_mul2(x, u) : silu_mul2(x, make_float2(1.0f, 1.0f));
        }
        out[i] = r.x;
        if (two) out[i + 1] = r.y;
    }
}

cudaError_t launch_debug_activation(int kind, const float* in, const float* in2, float* out, int64_t n,
                                    cudaStream_t stream) {
    const int64_t pairs = (n + 1) / 2;
    int64_t blocks = (pairs + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    debug_activation_kernel<<<(unsigned)blocks, 256, 0, stream>>>(kind, in, in2, out, n);
    return cudaGetLastError();
}
}  // namespace rmsq

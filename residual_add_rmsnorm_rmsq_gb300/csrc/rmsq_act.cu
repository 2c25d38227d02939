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

// The bounded mbarrier wait of the pipelined kernels, on a barrier that no
// copy and no thread ever completes: every thread must give up after
// `limit_ns` and the kernel must return normally, recording the outcome.
static __device__ int g_wait_outcome;
__global__ void debug_wait_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(&bar, 0u, limit_ns);
    const int gave_up = __syncthreads_count(!ok);
    if (threadIdx.x == 0) g_wait_outcome = gave_up == (int)blockDim.x ? 1 : (gave_up == 0 ? 0 : 2);
}

cudaError_t debug_bounded_wait(uint64_t limit_ns, int* outcome) {
    const int unset = -1;
    cudaError_t e = cudaMemcpyToSymbol(g_wait_outcome, &unset, sizeof(int));
    if (e != cudaSuccess) return e;
    debug_wait_kernel<<<1, 64>>>(limit_ns);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(outcome, g_wait_outcome, sizeof(int));
    return e;
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

// fp16 instantiations of the row kernel, and the conversion check kernel.
#include "rmsq_dispatch.cuh"

namespace rmsq {

// Same conversions as the kernels, one value per thread, for exhaustive checks.
__global__ void convert_kernel(int kind, const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float v = in[i];
        if (kind == 0) {
            out[i] = (uint8_t)(e4m3x2(v, 0.0f) & 0xffu);
        } else {
            float t[8] = {v, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            out[i] = (uint8_t)(e2m1x8(t) & 0xfu);
        }
    }
}

cudaError_t launch_rows_fp16(const LaunchArgs& a, cudaStream_t stream) {
    return launch_rows<Fp16T>(a, stream);
}

cudaError_t query_rows_fp16(const LaunchArgs& a, int* out) {
    RowLaunch l;
    const cudaError_t e = query_rows<Fp16T>(a, &l);
    if (e != cudaSuccess) return e;
    out[0] = l.pipe ? 1 : 0;
    out[1] = l.J;
    out[2] = l.stages;
    out[3] = l.grid;
    out[4] = l.threads;
    return cudaSuccess;
}

cudaError_t take_pipe_fault_fp16(unsigned int* out) { return take_pipe_fault(out); }

cudaError_t launch_nvfp4_dynamic_fp16(const LaunchArgs& a, void* workspace, float* out_gs, cudaStream_t stream) {
    return launch_nvfp4_dynamic<Fp16T>(a, workspace, out_gs, stream);
}

cudaError_t launch_convert(int kind, const float* in, uint8_t* out, int64_t n, cudaStream_t stream) {
    const int64_t blocks64 = (n + 255) / 256;
    const int blocks = (int)(blocks64 < 152 * 64 ? blocks64 : 152 * 64);
    convert_kernel<<<blocks, 256, 0, stream>>>(kind, in, out, n);
    return cudaGetLastError();
}
}  // namespace rmsq

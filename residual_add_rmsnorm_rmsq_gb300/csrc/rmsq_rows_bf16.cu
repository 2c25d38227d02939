// bf16 instantiations of the row kernel.
#include "rmsq_dispatch.cuh"

namespace rmsq {
cudaError_t launch_rows_bf16(const LaunchArgs& a, cudaStream_t stream) {
    return launch_rows<Bf16T>(a, stream);
}

cudaError_t query_rows_bf16(const LaunchArgs& a, int* out) {
    RowLaunch l;
    const cudaError_t e = query_rows<Bf16T>(a, &l);
    if (e != cudaSuccess) return e;
    out[0] = l.pipe ? 1 : 0;
    out[1] = l.J;
    out[2] = l.stages;
    out[3] = l.grid;
    out[4] = l.threads;
    return cudaSuccess;
}

cudaError_t take_pipe_fault_bf16(unsigned int* out) { return take_pipe_fault(out); }

cudaError_t launch_nvfp4_dynamic_bf16(const LaunchArgs& a, void* workspace, float* out_gs, cudaStream_t stream) {
    return launch_nvfp4_dynamic<Bf16T>(a, workspace, out_gs, stream);
}
}  // namespace rmsq

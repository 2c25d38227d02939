// bf16 instantiations of the row kernel.
#include "rmsq_dispatch.cuh"

namespace rmsq {
cudaError_t launch_rows_bf16(const LaunchArgs& a, cudaStream_t stream) {
    return launch_rows<Bf16T>(a, stream);
}

cudaError_t take_pipe_fault_bf16(unsigned int* out) { return take_pipe_fault(out); }

cudaError_t launch_nvfp4_dynamic_bf16(const LaunchArgs& a, void* workspace, float* out_gs, cudaStream_t stream) {
    return launch_nvfp4_dynamic<Bf16T>(a, workspace, out_gs, stream);
}
}  // namespace rmsq

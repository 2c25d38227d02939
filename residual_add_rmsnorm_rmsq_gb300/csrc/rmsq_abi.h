// Status helpers shared by the C ABI's translation units (not part of the
// public interface).
#pragma once

#include <cuda_runtime.h>

namespace rmsq_abi {

// Records `e` for rmsq_last_cuda_error() on this thread, clears it if it is
// not sticky, and returns RMSQ_ERR_CUDA.
int fail_cuda(cudaError_t e);

// RMSQ_OK when the current device is a compute capability 10.3 part;
// RMSQ_ERR_NO_DEVICE without a CUDA device, RMSQ_ERR_UNSUPPORTED_DEVICE for
// another one, RMSQ_ERR_CUDA (recorded) when the query itself fails.
int check_device();

}  // namespace rmsq_abi

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
    int variant;            // kVariant*
    bool e8m0;              // dynamic scales rounded up to a power of two
    bool ue8m0;             // ... and stored as one UE8M0 byte each
    int col_stride;         // column-major scale stride (n, or n rounded up to 16 bytes)
};

// LaunchArgs::mode of the norm alone (the kernels' Mode::kNormOnly).
constexpr int kModeNormOnly = 8;

constexpr int kVariantAuto = 0;
constexpr int kVariantDirect = 1;
constexpr int kVariantPipelined = 2;
// The pipelined kernel is chosen automatically from this many rows per SM.
constexpr int kPipeMinRowsPerSm = 4;

// Process-wide overrides of the pipelined launch shape (0 = automatic).
struct PipeTuning {
    int chunks_per_thread;
    int stages;
    int ctas_per_sm;
    int rows_per_iter;      // accepted for the API, unused: one row per CTA iteration
};
PipeTuning get_pipe_tuning();
void set_pipe_tuning(const PipeTuning& t);

// Whether the kernels are launched with programmatic stream serialisation
// (process-wide, on by default).
bool programmatic_launch();
void set_programmatic_launch(bool on);

// One launch of the row kernel for bf16 / fp16 activations.
cudaError_t launch_rows_bf16(const LaunchArgs& a, cudaStream_t stream);
cudaError_t launch_rows_fp16(const LaunchArgs& a, cudaStream_t stream);
// The launch launch_rows_* would make (none is made): out = {pipelined (0/1),
// chunks per thread, ring stages, CTAs, threads per CTA}.
cudaError_t query_rows_bf16(const LaunchArgs& a, int* out);
cudaError_t query_rows_fp16(const LaunchArgs& a, int* out);
// NVFP4 with a data-derived global scale (two passes); `workspace` holds the
// batch amax word and the per-row inv_rms.
cudaError_t launch_nvfp4_dynamic_bf16(const LaunchArgs& a, void* workspace, float* out_gs, cudaStream_t stream);
cudaError_t launch_nvfp4_dynamic_fp16(const LaunchArgs& a, void* workspace, float* out_gs, cudaStream_t stream);
// One CTA waits on an mbarrier nothing completes, bounded by limit_ns;
// *outcome: 1 every thread gave up, 0 none did, 2 some did.  Synchronous.
cudaError_t debug_bounded_wait(uint64_t limit_ns, int* outcome);
// The activation's e^x / silu / silu * u, elementwise (kind 0 / 1 / 2).
cudaError_t launch_debug_activation(int kind, const float* in, const float* in2, float* out, int64_t n,
                                    cudaStream_t stream);
// SiLU+Mul + quantisation: a.x = gate_up [n, 2d], a.hidden = d.
cudaError_t launch_act_bf16(const LaunchArgs& a, cudaStream_t stream);
cudaError_t launch_act_fp16(const LaunchArgs& a, cudaStream_t stream);
// Quantisation of a T tensor: a.x = [n, d], a.hidden = d.
cudaError_t launch_quant_bf16(const LaunchArgs& a, cudaStream_t stream);
cudaError_t launch_quant_fp16(const LaunchArgs& a, cudaStream_t stream);
// QK-norm + RoPE, in place on qkv.
struct QkLaunch {
    void* qkv;
    const int64_t* positions;
    const float* cos_sin;
    int64_t max_pos;
    const void* q_weight;
    const void* k_weight;
    float eps;
    int n, nq, nkv, head_dim;
    bool neox, fp16;
    int variant;   // kVariantAuto / kVariantDirect / kVariantPipelined
};
cudaError_t launch_qk_norm_rope(const QkLaunch& l, cudaStream_t stream);
// Workspace bytes for n rows (a 256-byte header, n fp32 inv_rms and at most n
// per-CTA partial maxima, rounded up to 256).
inline size_t nvfp4_dynamic_workspace_bytes(int64_t n) {
    const size_t raw = 256 + 8 * static_cast<size_t>(n);
    return (raw + 255) / 256 * 256;
}

// All-reduce + residual add + RMSNorm + quantisation: x is the rank-order
// fp32 sum of `n_ranks` partial buffers (la.x unused), rounded to T.
constexpr int kMaxArRanks = 8;
cudaError_t launch_allreduce_rows(const LaunchArgs& la, const void* const* partials, int n_ranks, bool fp16,
                                  cudaStream_t stream);

// Read and clear the pipelined kernels' fault flags (current device).
cudaError_t take_pipe_fault_bf16(unsigned int* out);
cudaError_t take_pipe_fault_fp16(unsigned int* out);
cudaError_t take_pipe_fault_qk(unsigned int* out);
cudaError_t take_pipe_fault_ar(unsigned int* out);
cudaError_t launch_convert(int kind, const float* in, uint8_t* out, int64_t n, cudaStream_t stream);

}  // namespace rmsq

// bf16 and fp16 instantiations of the QK-norm + RoPE kernels (warp and
// pipelined forms).
#include "rmsq_qk.cuh"

namespace rmsq {
cudaError_t launch_qk_norm_rope(const QkLaunch& l, cudaStream_t stream) {
    QkArgs a;
    a.qkv = static_cast<uint32_t*>(l.qkv);
    a.pos = l.positions;
    a.cs = l.cos_sin;
    a.max_pos = l.max_pos;
    a.qw = static_cast<const uint32_t*>(l.q_weight);
    a.kw = static_cast<const uint32_t*>(l.k_weight);
    a.eps = l.eps;
    a.inv_d = 1.0f / (float)l.head_dim;
    a.n = l.n;
    a.nq = l.nq;
    a.nkv = l.nkv;
    return l.fp16 ? launch_qk<Fp16T>(a, l.head_dim, l.neox, l.variant, stream)
                  : launch_qk<Bf16T>(a, l.head_dim, l.neox, l.variant, stream);
}
cudaError_t take_pipe_fault_qk(unsigned int* out) { return take_pipe_fault(out); }
}  // namespace rmsq

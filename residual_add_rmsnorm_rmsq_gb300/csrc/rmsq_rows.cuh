// Direct row kernel: one CTA per row, every load issued up front straight
// from global memory into registers.  Lowest latency for a handful of rows
// (decode batches); the pipelined kernel in rmsq_pipe.cuh takes over for
// batches that fill the GPU several times.
#pragma once

#include "rmsq_rowmath.cuh"

namespace rmsq {

template <class E, int MODE, bool RES, int J>
__global__ void __launch_bounds__(1024) rows_kernel(const RowArgs a) {
    __shared__ float s_sum[32];
    __shared__ float s_max[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row = blockIdx.x;
    const int64_t base = (int64_t)row * a.chunks;
    const int c0 = tid * J;

    uint4 xv[J], rv[J], wv[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        xv[j] = rv[j] = wv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (c0 + j < a.chunks) {
            xv[j] = ld_act(a.x + base + c0 + j);
            if constexpr (RES) rv[j] = ld_act(a.res + base + c0 + j);
            wv[j] = ld_weight(a.w + c0 + j);
        }
    }
    const float sin = ModeTraits<MODE>::needs_scale_in ? __ldg(a.scale_in) : 0.0f;

    float h[J][8];
    float acc = combine_chunks<E, RES, J>(xv, rv, h, a.res_out + base, c0, a.chunks);
    acc = warp_tree_sum(acc);
    if (lane == 0) s_sum[warp] = acc;
    __syncthreads();
    const float total = warp_tree_sum(lane < nwarps ? s_sum[lane] : 0.0f);
    const float inv = inv_rms(total, a.hidden, a.eps);
    quantize_row<E, MODE, J>(a, row, h, wv, inv, sin, s_max, tid, nwarps);
}

}  // namespace rmsq

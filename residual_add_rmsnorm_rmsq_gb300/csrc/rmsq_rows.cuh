// Direct row kernel: one CTA per row, every load issued up front straight
// from global memory into registers.  Lowest latency for a handful of rows
// (decode batches); the pipelined kernel in rmsq_pipe.cuh takes over for
// batches that fill the GPU several times.
#pragma once

#include "rmsq_rowmath.cuh"

namespace rmsq {

template <class E, int MODE, bool RES, int J>
__global__ void __launch_bounds__(1024) rows_kernel(const RowArgs a) {
    __shared__ __align__(16) float s_sum[32];
    __shared__ float s_max[32];
    // Slots of absent warps read as 0 (ordered before the reads by the barrier below).
    if (threadIdx.x < 32 && (int)threadIdx.x >= (int)(blockDim.x >> 5)) s_sum[threadIdx.x] = 0.0f;
    allow_dependents();
    grid_dependency_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row = blockIdx.x;
    const int64_t base = (int64_t)row * a.chunks;
    const int c0 = tid * J;

    uint4 xv[J], rv[J], wv[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        xv[j] = rv[j] = wv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (c0 + j < a.chunks) wv[j] = ld_weight(a.w + c0 + j);
    }
    if (J == 2 && a.pair) {   // chunks even: the pair is in the row or wholly past it
        if (c0 < a.chunks) {
            ld_act_pair(a.x + base + c0, xv[0], xv[J - 1]);
            if constexpr (RES) ld_act_pair(a.res + base + c0, rv[0], rv[J - 1]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (c0 + j < a.chunks) {
                xv[j] = ld_act(a.x + base + c0 + j);
                if constexpr (RES) rv[j] = ld_act(a.res + base + c0 + j);
            }
    }
    const float sin = ModeTraits<MODE>::needs_scale_in ? __ldg(a.scale_in) : 0.0f;
    __shared__ float s_rtab[MODE == kNvfp4 ? 128 : 1];
    if constexpr (MODE == kNvfp4) fill_nvfp4_rtab(s_rtab, sin);   // ordered by the barrier below

    uint32_t h[J][4];
    float acc = combine_chunks<E, RES, J, MODE == kNormAmax>(xv, rv, h, a.res_out + base, c0, a.chunks, a.pair);
    acc = warp_tree_sum(acc);
    if (lane == 0) s_sum[warp] = acc;
    __syncthreads();
    const float total = warp_slots_tree_sum<32>(s_sum, nwarps);
    const float inv = inv_rms(total, a);
    float run_max = 0.0f;
    float wf[J][8];
    widen_weights<E, J>(wv, wf);
    quantize_row<E, MODE, J>(a, row, h, wf, inv, sin, s_rtab, s_max, tid, nwarps, run_max);
    if constexpr (MODE == kNormAmax) flush_amax(a, run_max, s_max, tid, nwarps);
}

}  // namespace rmsq

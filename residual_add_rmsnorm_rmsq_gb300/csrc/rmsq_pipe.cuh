// Pipelined row kernel: persistent CTAs, each walking rows blockIdx.x,
// blockIdx.x + gridDim.x, ...; the x and residual rows of the next `stages`
// rows are in flight as bulk asynchronous copies (TMA, 1-D) into a ring of
// shared-memory stages while the current row is computed.  One elected thread
// issues the copies; a stage is refilled right after the CTA barrier that
// follows its last shared-memory read.  The weight row is loaded once into
// registers (every row of the launch uses it).
//
// Per row the arithmetic is the same as the direct kernel's (rmsq_rowmath.cuh):
// the canonical pairwise tree for the sum of squares, correctly rounded
// inverse RMS, fp32 y, then the quantisation mode.
//
// Every wait on a stage is bounded (mbar_wait_bounded).  If one ever gives up,
// the CTA records it in `fault`, drains the copies it still has in flight
// (again bounded) and returns.
#pragma once

#include "rmsq_rowmath.cuh"

namespace rmsq {

constexpr int kMaxStages = 8;
constexpr int kPipeMaxThreads = 512;

template <class E, int MODE, bool RES, int J>
__device__ __forceinline__ void pipe_body(const RowArgs& a, const int stages, unsigned int* fault) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ __align__(16) float s_sum[2][32];
    __shared__ float s_max[2][32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int c0 = tid * J;
    const int G = gridDim.x;
    const uint32_t row_bytes = static_cast<uint32_t>(a.chunks) * 16u;
    const uint32_t stage_bytes = RES ? 2u * row_bytes : row_bytes;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    if (tid < 64 && (tid & 31) >= nwarps) s_sum[tid >> 5][tid & 31] = 0.0f;   // absent warps: 0
    __syncthreads();

    uint64_t policy = 0;
    if (tid == 0) {
        policy = l2_policy_evict_first();
        for (int k = 0; k < stages; ++k) {
            const int row = blockIdx.x + k * G;
            if (row >= a.n) break;
            unsigned char* dst = ring + (size_t)k * stage_bytes;
            mbar_arrive_expect_tx(&full[k], stage_bytes);
            bulk_g2s(dst, a.x + (int64_t)row * a.chunks, row_bytes, &full[k], policy);
            if constexpr (RES)
                bulk_g2s(dst + row_bytes, a.res + (int64_t)row * a.chunks, row_bytes, &full[k], policy);
        }
    }

    uint4 wv[J];
#pragma unroll
    for (int j = 0; j < J; ++j)
        wv[j] = (c0 + j < a.chunks) ? ld_weight(a.w + c0 + j) : make_uint4(0u, 0u, 0u, 0u);
    const float sin = ModeTraits<MODE>::needs_scale_in ? __ldg(a.scale_in) : 0.0f;
    __shared__ float s_rtab[MODE == kNvfp4 ? 128 : 1];
    if constexpr (MODE == kNvfp4) fill_nvfp4_rtab(s_rtab, sin);   // ordered by the first row's barrier

    int k = 0;
    bool faulted = false;
    float run_max = 0.0f;
    for (;; ++k) {
        const int row = blockIdx.x + k * G;
        if (row >= a.n) break;
        const int s = k % stages;
        const uint32_t parity = static_cast<uint32_t>(k / stages) & 1u;
        const bool ok = mbar_wait_bounded(&full[s], parity);

        uint32_t h[J][4];
        float acc = 0.0f;
        if (ok) {
            const uint4* sx = reinterpret_cast<const uint4*>(ring + (size_t)s * stage_bytes);
            uint4 xv[J], rv[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                xv[j] = rv[j] = make_uint4(0u, 0u, 0u, 0u);
                if (c0 + j < a.chunks) {
                    xv[j] = sx[c0 + j];
                    if constexpr (RES) rv[j] = sx[a.chunks + c0 + j];
                }
            }
            acc = combine_chunks<E, RES, J>(xv, rv, h, a.res_out + (int64_t)row * a.chunks, c0, a.chunks);
        }
        acc = warp_tree_sum(acc);
        if (lane == 0) s_sum[k & 1][warp] = acc;
        // All reads of stage s are done once every thread is past this barrier.
        if (__syncthreads_or(!ok)) {
            faulted = true;
            break;
        }
        if (tid == 0) {
            const int nrow = row + stages * G;
            if (nrow < a.n) {
                unsigned char* dst = ring + (size_t)s * stage_bytes;
                mbar_arrive_expect_tx(&full[s], stage_bytes);
                bulk_g2s(dst, a.x + (int64_t)nrow * a.chunks, row_bytes, &full[s], policy);
                if constexpr (RES)
                    bulk_g2s(dst + row_bytes, a.res + (int64_t)nrow * a.chunks, row_bytes, &full[s], policy);
            }
        }
        const float total = smem_tree_sum<kPipeMaxThreads / 32>(s_sum[k & 1]);
        const float inv = inv_rms(total, a);
        quantize_row<E, MODE, J>(a, row, h, wv, inv, sin, s_rtab, s_max[k & 1], tid, nwarps, run_max);
    }
    if constexpr (MODE == kNormAmax) flush_amax(a, run_max, s_max[0], tid, nwarps);

    if (faulted && tid == 0) {
        atomicOr(fault, 1u);
        // Copies issued for rows k .. k + stages - 1 may still be in flight.
        for (int kk = k; kk < k + stages; ++kk) {
            if (blockIdx.x + kk * G >= a.n) break;
            mbar_wait_bounded(&full[kk % stages], static_cast<uint32_t>(kk / stages) & 1u);
        }
    }
}

}  // namespace rmsq

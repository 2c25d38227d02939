// Pipelined row kernel: persistent CTAs, each walking groups of R rows
// (rows blockIdx.x + (k*R + r) * gridDim.x for r < R); the x and residual rows
// of the next `stages` groups are in flight as bulk asynchronous copies (TMA,
// 1-D) into a ring of shared-memory stages while the current group is
// computed.  One elected thread issues the copies; a stage is refilled right
// after the CTA barrier that follows its last shared-memory read.  The weight
// row is loaded once into registers (every row of the launch uses it).
//
// R = 2 interleaves two rows: their reductions share each CTA barrier, so the
// latency of the per-row dependency chain (block reductions, IEEE divide and
// square root) is paid once per two rows.
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

template <class E, int MODE, bool RES, int J, int R>
__device__ __forceinline__ void pipe_body(const RowArgs& a, const int stages, unsigned int* fault) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ __align__(16) float s_sum[2][R][32];
    __shared__ float s_max[2][R][32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int c0 = tid * J;
    const int G = gridDim.x;
    const uint32_t row_bytes = static_cast<uint32_t>(a.chunks) * 16u;
    const uint32_t slot_bytes = RES ? 2u * row_bytes : row_bytes;   // one row of x (+ residual)
    const uint32_t stage_bytes = R * slot_bytes;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    // Slots of absent warps read as 0, in both halves of the double buffer and
    // for every row of a group, whatever the CTA size (a one-warp CTA has
    // only 32 threads to clear 2 * R * 31 slots).
    for (int i = tid; i < 2 * R * 32; i += blockDim.x)
        if ((i & 31) >= nwarps) (&s_sum[0][0][0])[i] = 0.0f;
    allow_dependents();
    grid_dependency_wait();
    __syncthreads();

    // Thread 0: start the copies of row group k into stage s.
    uint64_t policy = 0;
    auto issue = [&](int k, int s) {
        unsigned char* dst = ring + (size_t)s * stage_bytes;
        uint32_t bytes = 0;
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (blockIdx.x + (k * R + r) * G < a.n) bytes += slot_bytes;
        mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = blockIdx.x + (k * R + r) * G;
            if (row >= a.n) break;
            bulk_g2s(dst + r * slot_bytes, a.x + (int64_t)row * a.chunks, row_bytes, &full[s], policy);
            if constexpr (RES)
                bulk_g2s(dst + r * slot_bytes + row_bytes, a.res + (int64_t)row * a.chunks, row_bytes,
                         &full[s], policy);
        }
    };
    // The first pass of the data-derived NVFP4 scale is followed by a pass
    // that reads h again: without a residual h is x, kept in L2.
    constexpr bool KEEP = MODE == kNormAmax;
    if (tid == 0) {
        policy = (KEEP && !RES) ? l2_policy_evict_normal() : l2_policy_evict_first();
        for (int k = 0; k < stages; ++k) {
            if (blockIdx.x + k * R * G >= a.n) break;
            issue(k, k);
        }
    }

    float wv[J][8];
    {
        uint4 wraw[J];
#pragma unroll
        for (int j = 0; j < J; ++j)
            wraw[j] = (c0 + j < a.chunks) ? ld_weight(a.w + c0 + j) : make_uint4(0u, 0u, 0u, 0u);
        widen_weights<E, J>(wraw, wv);
    }
    const float sin = ModeTraits<MODE>::needs_scale_in ? __ldg(a.scale_in) : 0.0f;
    __shared__ float s_rtab[MODE == kNvfp4 ? 128 : 1];
    if constexpr (MODE == kNvfp4) fill_nvfp4_rtab(s_rtab, sin);   // ordered by the first barrier

    int k = 0;
    bool faulted = false;
    float run_max = 0.0f;
    for (;; ++k) {
        const int row0 = blockIdx.x + k * R * G;
        if (row0 >= a.n) break;
        const int s = k % stages;
        const uint32_t parity = static_cast<uint32_t>(k / stages) & 1u;
        const bool ok = mbar_wait_bounded(&full[s], parity);

        uint32_t hw[R][J][4];
        float acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = row0 + r * G;
            acc[r] = 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j) hw[r][j][0] = hw[r][j][1] = hw[r][j][2] = hw[r][j][3] = 0u;
            if (ok && row < a.n) {
                const uint4* sx =
                    reinterpret_cast<const uint4*>(ring + (size_t)s * stage_bytes + (size_t)r * slot_bytes);
                uint4 xv[J], rv[J];
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    xv[j] = rv[j] = make_uint4(0u, 0u, 0u, 0u);
                    if (c0 + j < a.chunks) {
                        xv[j] = sx[c0 + j];
                        if constexpr (RES) rv[j] = sx[a.chunks + c0 + j];
                    }
                }
                acc[r] = combine_chunks<E, RES, J, KEEP>(xv, rv, hw[r], a.res_out + (int64_t)row * a.chunks,
                                                         c0, a.chunks, a.pair);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            acc[r] = warp_tree_sum(acc[r]);
            if (lane == 0) s_sum[k & 1][r][warp] = acc[r];
        }
        // All reads of stage s are done once every thread is past this barrier.
        if (__syncthreads_or(!ok)) {
            faulted = true;
            break;
        }
        if (tid == 0 && blockIdx.x + (k + stages) * R * G < a.n) issue(k + stages, s);

        float inv[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            inv[r] = inv_rms(warp_slots_tree_sum<kPipeMaxThreads / 32>(s_sum[k & 1][r], nwarps), a);

        if constexpr (MODE == kFp8PerToken && R > 1) {
            // The rows' amax reductions share one barrier.
            float y[R][J][8];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                compute_y<E, J>(hw[r], wv, inv[r], y[r]);
                per_token_warp_amax<J>(y[r], s_max[k & 1][r], lane, warp);
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (row0 + r * G < a.n)
                    per_token_finish<J>(a, row0 + r * G, y[r], s_max[k & 1][r], tid, nwarps);
        } else {
            // No barrier inside quantize_row for these modes (per-token only with R == 1,
            // where every thread takes the r == 0 call).
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (r == 0 || row0 + r * G < a.n)
                    quantize_row<E, MODE, J>(a, row0 + r * G, hw[r], wv, inv[r], sin, s_rtab, s_max[k & 1][r],
                                             tid, nwarps, run_max);
        }
    }
    if constexpr (MODE == kNormAmax) flush_amax(a, run_max, s_max[0][0], tid, nwarps);

    if (faulted && tid == 0) {
        atomicOr(fault, 1u);
        // Copies issued for row groups k .. k + stages - 1 may still be in flight.
        for (int kk = k; kk < k + stages; ++kk) {
            if (blockIdx.x + kk * R * G >= a.n) break;
            mbar_wait_bounded(&full[kk % stages], static_cast<uint32_t>(kk / stages) & 1u);
        }
    }
}

}  // namespace rmsq

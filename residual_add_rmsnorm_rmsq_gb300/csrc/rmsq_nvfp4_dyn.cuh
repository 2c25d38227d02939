// NVFP4 with the global scale taken from the data (gs = 448 * 6 / amax of y
// over the whole batch, 1 for an all-zero batch), in two passes:
//
//  1. the row work in mode kNormAmax: residual add and write-back, RMSNorm,
//     the row's inv_rms into the workspace, and each CTA's amax of |y| into
//     its slot of the workspace;
//  2. nvfp4_dyn_column below: each thread owns one column of 16-element
//     blocks, re-reads h (residual_out, or x without a residual) over its
//     rows, rebuilds y = (h * inv) * w exactly as pass 1 did, and writes the
//     E4M3 block scale and the eight bytes of E2M1 codes with
//     gs = 2688 / amax, amax being the max of pass 1's per-CTA slots.
//
// Two launches and no atomics: the workspace needs no zeroing, so its
// contents on entry do not matter.
//
// Pass 1 stores h at normal L2 priority (not streaming), so that pass 2,
// launched right after it, finds a small batch's h in L2; tens of MB of h
// (16384 rows of 2048) come back from DRAM all the same.
//
// The NVFP4 step follows the vLLM PR #51925 summary ("Motivation": block
// scales and FP4 values from the normalised activations and an fp32 global
// scale); the rule for gs is the NVFP4 workload's definition.
#pragma once

#include "rmsq_rowmath.cuh"

namespace rmsq {

// E4M3 block scale of 16 values y under global scale gs, and their E2M1
// codes (element k in nibble k of the 8 bytes).  The products y * r are
// formed in packed pairs (y[k], y[8 + k]).
__device__ __forceinline__ uint32_t nvfp4_block16(const float (&y)[16], float gs, const float* rtab,
                                                  uint2& codes) {
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; k += 2) m = max_abs3(m, y[k], y[k + 1]);
    const uint32_t sb = e4m3x2(__fmul_rn(__fdiv_rn(m, 6.0f), gs), 0.0f) & 0xffu;
    const float r = rtab[sb];      // gs / decode(sb), 0 for a zero block scale
    float lo[8], hi[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 t = mul2_rn(make_float2(y[k], y[8 + k]), make_float2(r, r));
        lo[k] = t.x;
        hi[k] = t.y;
    }
    codes.x = e2m1x8(lo);
    codes.y = e2m1x8(hi);
    return sb;
}

// Rows of a pass-2 thread's column loaded before any is computed
// (compile-time tuning; results do not depend on it).
#ifndef RMSQ_DYN_ROWS
#define RMSQ_DYN_ROWS 2
#endif
constexpr int kDynRows = RMSQ_DYN_ROWS;

// Pass 2 for one column of 16-element blocks: thread t of the R * bpr
// threads (bpr = hidden / 16 blocks per row) takes block column
// cb = t mod bpr of the rows t / bpr, t / bpr + R, t / bpr + 2R, ...  Its
// weights are loaded and widened once, and the rows advance by a constant
// stride, so the loop carries no index division.  y = (h * inv) * w is
// rebuilt exactly as pass 1 formed it (same roundings; the packed pairs here
// are element k of the block's two chunks), then the block scale and codes
// under gs.  `pair`: h starts on 32 bytes, so a block's two chunks are one
// load.
template <class E>
__device__ __forceinline__ void nvfp4_dyn_column(const uint4* h, const uint4* w, const float* ws, uint2* q,
                                                 uint8_t* bscale, int n, int hidden, float gs,
                                                 const float* rtab, int t, int R, bool pair) {
    const int bpr = hidden / 16;
    const int chunks = hidden / 8;
    const int cb = t % bpr;
    const int r0 = t / bpr;
    if (r0 >= n) return;
    const uint4 wa = ld_weight(w + 2 * cb), wb = ld_weight(w + 2 * cb + 1);
    const uint32_t w0[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t w1[4] = {wb.x, wb.y, wb.z, wb.w};
    float2 wlo[4], whi[4];   // (w[2k], w[8 + 2k]) and (w[2k + 1], w[8 + 2k + 1])
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        wlo[k] = make_float2(E::lo(w0[k]), E::lo(w1[k]));
        whi[k] = make_float2(E::hi(w0[k]), E::hi(w1[k]));
    }
    const int64_t hstep = (int64_t)R * chunks;
    const int64_t bstep = (int64_t)R * bpr;
    const uint4* hp = h + (int64_t)r0 * chunks + 2 * cb;
    uint2* qp = q + (int64_t)r0 * bpr + cb;
    uint8_t* sp = bscale + (int64_t)r0 * bpr + cb;
    const float* ip = ws + kWsInvOffset + r0;
    // The thread's rows: r0, r0 + R, ... below n (m of them), kDynRows per
    // iteration with all their loads issued first.
    const int m = (n - 1 - r0) / R + 1;
    for (int i = 0; i < m; i += kDynRows) {
        uint4 hv[kDynRows][2];
        float inv[kDynRows];
#pragma unroll
        for (int u = 0; u < kDynRows; ++u) {
            if (i + u < m) {
                const uint4* p = hp + u * hstep;
                inv[u] = ip[(int64_t)u * R];
                if (pair) {
                    ld_act_pair(p, hv[u][0], hv[u][1]);
                } else {
                    hv[u][0] = ld_act(p);
                    hv[u][1] = ld_act(p + 1);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kDynRows; ++u) {
            if (i + u >= m) break;
            const uint32_t h0[4] = {hv[u][0].x, hv[u][0].y, hv[u][0].z, hv[u][0].w};
            const uint32_t h1[4] = {hv[u][1].x, hv[u][1].y, hv[u][1].z, hv[u][1].w};
            const float2 iv = make_float2(inv[u], inv[u]);
            float y[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 a = mul2_rn(mul2_rn(make_float2(E::lo(h0[k]), E::lo(h1[k])), iv), wlo[k]);
                const float2 c = mul2_rn(mul2_rn(make_float2(E::hi(h0[k]), E::hi(h1[k])), iv), whi[k]);
                y[2 * k] = a.x; y[8 + 2 * k] = a.y;
                y[2 * k + 1] = c.x; y[8 + 2 * k + 1] = c.y;
            }
            uint2 codes;
            const uint32_t sb = nvfp4_block16(y, gs, rtab, codes);
            st_stream(qp + u * bstep, codes);
            sp[u * bstep] = (uint8_t)sb;
        }
        hp += kDynRows * hstep;
        qp += kDynRows * bstep;
        sp += kDynRows * bstep;
        ip += (int64_t)kDynRows * R;
    }
}

// 256-thread CTAs per SM that pass 2 is sized for (compile-time tuning; 0:
// as many as are resident at once, so each thread walks its column through
// all its rows in one pass of the grid).
#ifndef RMSQ_DYN_CTAS_PER_SM
#define RMSQ_DYN_CTAS_PER_SM 0
#endif
constexpr int kDynCtasPerSm = RMSQ_DYN_CTAS_PER_SM;

// Threads of pass 2 for n rows of `hidden` (R rows per sweep, R * bpr
// threads), about `target` threads in all.
inline void nvfp4_dyn_shape(int n, int hidden, int64_t target, int* rows_per_sweep, int* threads) {
    const int64_t bpr = hidden / 16;
    int64_t R = target / bpr;
    if (R < 1) R = 1;
    if (R > n) R = n > 0 ? n : 1;
    *rows_per_sweep = (int)R;
    *threads = (int)(R * bpr);
}

// gs = 2688 / amax, 1 when the batch amax is 0.
__device__ __forceinline__ float nvfp4_dyn_gs(float amax) { return amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f; }

// Pass 2 as its own kernel, launched after pass 1: the batch amax is the max
// of pass 1's `parts` per-CTA partial maxima (a few KB, read from L2 by every
// CTA; non-negative floats order like their bit patterns), then gs and the
// blocks.
template <class E>
__global__ void __launch_bounds__(256) nvfp4_dyn_quant_kernel(const uint4* h, const uint4* w,
                                                              const float* ws, uint2* q,
                                                              uint8_t* bscale, float* out_gs,
                                                              int n, int hidden, int pair, int parts,
                                                              int rows_per_sweep, int threads) {
    __shared__ float s_rtab[128];
    __shared__ unsigned int s_max[8];
    allow_dependents();
    grid_dependency_wait();
    const unsigned int* slots = reinterpret_cast<const unsigned int*>(ws + kWsInvOffset + n);
    // Eight independent loads in flight per thread and round (2048 slots per
    // round for 256 threads), so the slots cost one L2 round trip, not one per
    // iteration.
    unsigned int m = 0u;
    for (int base = 0; base < parts; base += 8 * (int)blockDim.x) {
        unsigned int v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + u * (int)blockDim.x + (int)threadIdx.x;
            v[u] = i < parts ? __ldcg(slots + i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) m = max(m, v[u]);
    }
    m = __reduce_max_sync(kFull, m);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0u;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = max(m, s_max[i]);
    const float gs = nvfp4_dyn_gs(__uint_as_float(m));
    if (blockIdx.x == 0 && threadIdx.x == 0) *out_gs = gs;
    fill_nvfp4_rtab(s_rtab, gs);
    __syncthreads();
    const int t = (int)(blockIdx.x * blockDim.x + threadIdx.x);
    if (t < threads)
        nvfp4_dyn_column<E>(h, w, ws, q, bscale, n, hidden, gs, s_rtab, t, rows_per_sweep, pair != 0);
}

}  // namespace rmsq

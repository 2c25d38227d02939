// NVFP4 with the global scale taken from the data (gs = 448 * 6 / amax of y
// over the whole batch, 1 for an all-zero batch), in two passes:
//
//  1. the row work in mode kNormAmax: residual add and write-back, RMSNorm,
//     the row's inv_rms into the workspace, and each CTA's amax of |y| into
//     its slot of the workspace;
//  2. nvfp4_dyn_blocks below: one thread per 16-element block re-reads h
//     (residual_out, or x without a residual) and the weight, rebuilds
//     y = (h * inv) * w exactly as pass 1 did, and writes the E4M3 block
//     scale and the eight bytes of E2M1 codes with gs = 2688 / amax, amax
//     being the max of pass 1's per-CTA slots.
//
// Two launches and no atomics: the workspace needs no zeroing, so its
// contents on entry do not matter.
//
// Pass 1 keeps h at normal L2 priority, so that pass 2, launched right after
// it, mostly reads h from L2.
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

// Blocks of 16 each thread of pass 2 loads before computing (compile-time
// tuning; results do not depend on it).
#ifndef RMSQ_DYN_UNROLL
#define RMSQ_DYN_UNROLL 1
#endif
constexpr int kDynUnroll = RMSQ_DYN_UNROLL;

// Pass 2 over the 16-element blocks first, first + stride, ... of the n x
// hidden/16 blocks: y = (h * inv) * w rebuilt exactly as pass 1 formed it
// (same roundings; the packed pairs here are element k of the block's two
// chunks), then the block scale and codes under gs.
// `pair`: h and w start on 32 bytes, so a block's two chunks are one load.
template <class E>
__device__ __forceinline__ void nvfp4_dyn_blocks(const uint4* h, const uint4* w, const float* ws, uint2* q,
                                                 uint8_t* bscale, int n, int hidden, float gs,
                                                 const float* rtab, int64_t first, int64_t stride, bool pair) {
    const int bpr = hidden / 16;
    const int chunks = hidden / 8;
    const int64_t total = (int64_t)n * bpr;
    // kDynUnroll blocks per thread and iteration, all loads issued first.
    for (int64_t b0 = first; b0 < total; b0 += kDynUnroll * stride) {
        uint4 hv[kDynUnroll][2], wv[kDynUnroll][2];
        float inv[kDynUnroll];
#pragma unroll
        for (int u = 0; u < kDynUnroll; ++u) {
            const int64_t b = b0 + u * stride;
            if (b < total) {
                const int row = (int)(b / bpr);
                const int cb = (int)(b - (int64_t)row * bpr);
                const uint4* hp = h + (int64_t)row * chunks + 2 * cb;
                inv[u] = ws[kWsInvOffset + row];
                if (pair) {
                    ld_act_pair(hp, hv[u][0], hv[u][1]);
                } else {
                    hv[u][0] = ld_act(hp);
                    hv[u][1] = ld_act(hp + 1);
                }
                wv[u][0] = ld_weight(w + 2 * cb);
                wv[u][1] = ld_weight(w + 2 * cb + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < kDynUnroll; ++u) {
            const int64_t b = b0 + u * stride;
            if (b >= total) break;
            const uint32_t h0[4] = {hv[u][0].x, hv[u][0].y, hv[u][0].z, hv[u][0].w};
            const uint32_t h1[4] = {hv[u][1].x, hv[u][1].y, hv[u][1].z, hv[u][1].w};
            const uint32_t w0[4] = {wv[u][0].x, wv[u][0].y, wv[u][0].z, wv[u][0].w};
            const uint32_t w1[4] = {wv[u][1].x, wv[u][1].y, wv[u][1].z, wv[u][1].w};
            const float2 iv = make_float2(inv[u], inv[u]);
            float y[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 a = mul2_rn(mul2_rn(make_float2(E::lo(h0[k]), E::lo(h1[k])), iv),
                                         make_float2(E::lo(w0[k]), E::lo(w1[k])));
                const float2 c = mul2_rn(mul2_rn(make_float2(E::hi(h0[k]), E::hi(h1[k])), iv),
                                         make_float2(E::hi(w0[k]), E::hi(w1[k])));
                y[2 * k] = a.x; y[8 + 2 * k] = a.y;
                y[2 * k + 1] = c.x; y[8 + 2 * k + 1] = c.y;
            }
            uint2 codes;
            const uint32_t sb = nvfp4_block16(y, gs, rtab, codes);
            st_stream(q + b, codes);
            bscale[b] = (uint8_t)sb;
        }
    }
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
                                                              int n, int hidden, int pair, int parts) {
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
    nvfp4_dyn_blocks<E>(h, w, ws, q, bscale, n, hidden, gs, s_rtab,
                               (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                               (int64_t)gridDim.x * blockDim.x, pair != 0);
}

}  // namespace rmsq

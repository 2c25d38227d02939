// NVFP4 with the global scale taken from the data (gs = 448 * 6 / amax of y
// over the whole batch, 1 for an all-zero batch), in two passes:
//
//  1. the row kernels in mode kNormAmax: residual add and write-back,
//     RMSNorm, the row's inv_rms into the workspace, and the batch amax of |y|
//     (one atomicMax per CTA on the workspace's amax word, zeroed before);
//  2. nvfp4_dyn_quant_kernel below: one thread per 16-element block re-reads
//     h (residual_out, or x without a residual) and the weight, rebuilds
//     y = (h * inv) * w exactly as pass 1 did, and writes the E4M3 block
//     scale and the eight bytes of E2M1 codes with gs = 2688 / amax.
//
// The NVFP4 step follows the vLLM PR #51925 summary ("Motivation": block
// scales and FP4 values from the normalised activations and an fp32 global
// scale); the rule for gs is the NVFP4 workload's definition.
#pragma once

#include "rmsq_rowmath.cuh"

namespace rmsq {

// E4M3 block scale of 16 values y under global scale gs, and their E2M1
// codes (element k in nibble k of the 8 bytes).
__device__ __forceinline__ uint32_t nvfp4_block16(const float (&y)[16], float gs, const float* rtab,
                                                  uint2& codes) {
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) m = fmaxf(m, fabsf(y[k]));
    const uint32_t sb = e4m3x2(__fmul_rn(__fdiv_rn(m, 6.0f), gs), 0.0f) & 0xffu;
    const float r = rtab[sb];      // gs / decode(sb), 0 for a zero block scale
    float lo[8], hi[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        lo[k] = __fmul_rn(y[k], r);
        hi[k] = __fmul_rn(y[8 + k], r);
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

template <class E>
__global__ void __launch_bounds__(256) nvfp4_dyn_quant_kernel(const uint4* h, const uint4* w,
                                                              const float* ws, uint2* q,
                                                              uint8_t* bscale, float* out_gs,
                                                              int n, int hidden) {
    allow_dependents();
    grid_dependency_wait();
    const float amax = __uint_as_float(reinterpret_cast<const unsigned int*>(ws)[0]);
    const float gs = amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *out_gs = gs;
    __shared__ float s_rtab[128];
    fill_nvfp4_rtab(s_rtab, gs);
    __syncthreads();
    const int bpr = hidden / 16;
    const int chunks = hidden / 8;
    const int64_t total = (int64_t)n * bpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // kDynUnroll blocks per thread and iteration, all loads issued first.
    for (int64_t b0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b0 < total;
         b0 += kDynUnroll * stride) {
        uint4 hv[kDynUnroll][2], wv[kDynUnroll][2];
        float inv[kDynUnroll];
#pragma unroll
        for (int u = 0; u < kDynUnroll; ++u) {
            const int64_t b = b0 + u * stride;
            if (b < total) {
                const int row = (int)(b / bpr);
                const int cb = (int)(b - (int64_t)row * bpr);
                inv[u] = ws[kWsInvOffset + row];
                hv[u][0] = ld_act(h + (int64_t)row * chunks + 2 * cb);
                hv[u][1] = ld_act(h + (int64_t)row * chunks + 2 * cb + 1);
                wv[u][0] = ld_weight(w + 2 * cb);
                wv[u][1] = ld_weight(w + 2 * cb + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < kDynUnroll; ++u) {
            const int64_t b = b0 + u * stride;
            if (b >= total) break;
            float y[16];
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const uint32_t hs[4] = {hv[u][v].x, hv[u][v].y, hv[u][v].z, hv[u][v].w};
                const uint32_t wsv[4] = {wv[u][v].x, wv[u][v].y, wv[u][v].z, wv[u][v].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    y[8 * v + 2 * k] = __fmul_rn(__fmul_rn(E::lo(hs[k]), inv[u]), E::lo(wsv[k]));
                    y[8 * v + 2 * k + 1] = __fmul_rn(__fmul_rn(E::hi(hs[k]), inv[u]), E::hi(wsv[k]));
                }
            }
            uint2 codes;
            const uint32_t sb = nvfp4_block16(y, gs, s_rtab, codes);
            st_stream(q + b, codes);
            bscale[b] = (uint8_t)sb;
        }
    }
}

}  // namespace rmsq

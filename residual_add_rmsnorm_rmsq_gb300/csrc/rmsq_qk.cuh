// QK-norm + RoPE (vLLM docs "Fusion torch.compile passes", section "QK Norm +
// RoPE (enable_qk_norm_rope_fusion)": split QKV, per-head RMSNorm of Q and K,
// rotary position embedding, in one kernel), in place on qkv.
//
// A warp works on 32 * 16 / head_dim heads of one token at a time; lane g of
// a head holds its elements 16g .. 16g+15, so the head's sum of squares is
// the canonical pairwise tree (in-lane tree, then the xor butterfly over the
// head's lanes) and the norm is the norm op's (inv = 1 / sqrt(S / D + eps),
// y = (x * inv) * w, fp32).  RoPE rotates pairs with cos / sin read from the
// caller's fp32 table at the token's position: NeoX pairs element i with
// i + D/2 (lanes g and g + D/32), GPT-J pairs 2i with 2i + 1 (inside a lane);
// every product and sum is rounded separately and the result is rounded once
// to the activation type.  v heads are not touched; a token whose position is
// outside [0, max_pos) is left unchanged.
#pragma once

#include "rmsq_dispatch.cuh"

namespace rmsq {

struct QkArgs {
    uint32_t* qkv;            // [n, (nq + 2 nkv) D] T, as 32-bit words
    const int64_t* pos;       // [n]
    const float* cs;          // [max_pos, D]: cos (D/2), sin (D/2)
    int64_t max_pos;
    const uint32_t* qw;       // [D] T
    const uint32_t* kw;       // [D] T
    float eps;
    float inv_d;              // 1 / D (exact: D is a power of two)
    int n, nq, nkv;
};

template <int EPL>
__device__ __forceinline__ float lane_leaf_sumsq(const float (&x)[EPL]) {
    float v[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) v[i] = __fmul_rn(x[i], x[i]);
#pragma unroll
    for (int len = EPL; len > 1; len >>= 1)
#pragma unroll
        for (int k = 0; k < len / 2; ++k) v[k] = __fadd_rn(v[2 * k], v[2 * k + 1]);
    return v[0];
}

// Elements per lane: a head of D elements takes D / 16 lanes (4, 8 or 16),
// so one warp works on 32 * 16 / D heads of a token together and shares the
// per-head scalar work (butterfly, square root, division) across them.
constexpr int kQkEpl = 16;

// Resident 256-thread CTAs per SM the kernel is compiled for (the register
// budget follows from it); compile-time tuning, results do not depend on it.
// Tighter budgets spill and were slower on GB300.
#ifndef RMSQ_QK_MIN_BLOCKS
#define RMSQ_QK_MIN_BLOCKS 1
#endif

template <class E, int D, bool NEOX>
__global__ void __launch_bounds__(256, RMSQ_QK_MIN_BLOCKS) qk_norm_rope_kernel(const QkArgs a) {
    constexpr int EPL = kQkEpl, W = EPL / 2;    // elements and 32-bit words per lane
    static_assert(W == 8, "two 16-byte accesses per lane");
    constexpr int LPH = D / EPL;                // lanes per head
    constexpr int HPW = 32 / LPH;               // heads per warp
    constexpr int NCS = NEOX ? EPL : EPL / 2;   // angles per lane
    allow_dependents();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int g = lane % LPH, r = lane / LPH;   // lane within its head, head within the warp
    const int heads = a.nq + a.nkv;
    const int chunks = (heads + HPW - 1) / HPW;  // warps per token
    const int width_words = (heads + a.nkv) * D / 2;
    const int total = a.n * chunks;
    const int step = gridDim.x * (blockDim.x >> 5);
    for (int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += step) {
        const int t = w / chunks;
        const int hd = (w - t * chunks) * HPW + r;
        const int64_t p = __ldg(a.pos + t);
        if (p < 0 || p >= a.max_pos) continue;   // the same for the whole warp
        const bool live = hd < heads;
        // loads first: the head's elements, its weight, the token's cos / sin
        uint32_t xw[W] = {}, ww[W] = {};
        uint4* hp = reinterpret_cast<uint4*>(a.qkv + (int64_t)t * width_words + hd * (D / 2) + g * W);
        if (live) {
            const uint4 x0 = ld_act(hp), x1 = ld_act(hp + 1);
            const uint4* wp = reinterpret_cast<const uint4*>((hd < a.nq ? a.qw : a.kw) + g * W);
            const uint4 w0 = __ldg(wp), w1 = __ldg(wp + 1);
            xw[0] = x0.x; xw[1] = x0.y; xw[2] = x0.z; xw[3] = x0.w;
            xw[4] = x1.x; xw[5] = x1.y; xw[6] = x1.z; xw[7] = x1.w;
            ww[0] = w0.x; ww[1] = w0.y; ww[2] = w0.z; ww[3] = w0.w;
            ww[4] = w1.x; ww[5] = w1.y; ww[6] = w1.z; ww[7] = w1.w;
        }
        float cv[NCS], sv[NCS];
        {
            const float4* cs = reinterpret_cast<const float4*>(a.cs + p * D + (NEOX ? (g % (LPH / 2)) * EPL : g * EPL / 2));
#pragma unroll
            for (int k = 0; k < NCS / 4; ++k) {
                const float4 c = __ldg(cs + k), s4 = __ldg(cs + D / 8 + k);
                cv[4 * k] = c.x; cv[4 * k + 1] = c.y; cv[4 * k + 2] = c.z; cv[4 * k + 3] = c.w;
                sv[4 * k] = s4.x; sv[4 * k + 1] = s4.y; sv[4 * k + 2] = s4.z; sv[4 * k + 3] = s4.w;
            }
        }
        float x[EPL], y[EPL];
#pragma unroll
        for (int i = 0; i < W; ++i) { x[2 * i] = E::lo(xw[i]); x[2 * i + 1] = E::hi(xw[i]); }
        // the head's sum: in-lane tree, then the butterfly over its LPH lanes
        float sum = lane_leaf_sumsq<EPL>(x);
#pragma unroll
        for (int o = 1; o < LPH; o <<= 1) sum = __fadd_rn(sum, __shfl_xor_sync(kFull, sum, o));
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(sum, a.inv_d), a.eps)));
#pragma unroll
        for (int i = 0; i < W; ++i) {
            y[2 * i] = __fmul_rn(__fmul_rn(x[2 * i], inv), E::lo(ww[i]));
            y[2 * i + 1] = __fmul_rn(__fmul_rn(x[2 * i + 1], inv), E::hi(ww[i]));
        }
        float o[EPL];
        if constexpr (NEOX) {
            // lanes g < LPH/2 hold the first halves a (element i), the others the
            // second halves b (element i + D/2); angle index (g mod LPH/2) * EPL + k
            const bool first = g < LPH / 2;
#pragma unroll
            for (int k = 0; k < EPL; ++k) {
                const float partner = __shfl_xor_sync(kFull, y[k], LPH / 2);
                o[k] = first ? __fsub_rn(__fmul_rn(y[k], cv[k]), __fmul_rn(partner, sv[k]))    // a c - b s
                             : __fadd_rn(__fmul_rn(y[k], cv[k]), __fmul_rn(partner, sv[k]));   // b c + a s
            }
        } else {
#pragma unroll
            for (int m = 0; m < EPL / 2; ++m) {
                const float ya = y[2 * m], yb = y[2 * m + 1];
                o[2 * m] = __fsub_rn(__fmul_rn(ya, cv[m]), __fmul_rn(yb, sv[m]));
                o[2 * m + 1] = __fadd_rn(__fmul_rn(yb, cv[m]), __fmul_rn(ya, sv[m]));
            }
        }
        if (live) {
            uint32_t ow[W];
#pragma unroll
            for (int i = 0; i < W; ++i) ow[i] = E::pack(o[2 * i], o[2 * i + 1]);
            st_stream(hp, make_uint4(ow[0], ow[1], ow[2], ow[3]));
            st_stream(hp + 1, make_uint4(ow[4], ow[5], ow[6], ow[7]));
        }
    }
}

template <class E>
cudaError_t launch_qk(const QkArgs& a, int head_dim, bool neox, cudaStream_t stream) {
    const void* fn = nullptr;
    switch (head_dim) {
    case 64: fn = neox ? (const void*)&qk_norm_rope_kernel<E, 64, true> : (const void*)&qk_norm_rope_kernel<E, 64, false>; break;
    case 128: fn = neox ? (const void*)&qk_norm_rope_kernel<E, 128, true> : (const void*)&qk_norm_rope_kernel<E, 128, false>; break;
    case 256: fn = neox ? (const void*)&qk_norm_rope_kernel<E, 256, true> : (const void*)&qk_norm_rope_kernel<E, 256, false>; break;
    default: return cudaErrorInvalidValue;
    }
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (err != cudaSuccess) return err;
    const int hpw = 32 * kQkEpl / head_dim;
    const int64_t warps = (int64_t)a.n * ((a.nq + a.nkv + hpw - 1) / hpw);
    int64_t grid = (warps + 7) / 8;
    if (grid > (int64_t)sms * 32) grid = (int64_t)sms * 32;
    QkArgs args = a;
    void* params[] = {&args};
    return launch_kernel(fn, dim3((unsigned)grid), dim3(256), params, 0, stream);
}

}  // namespace rmsq

// Row kernel of the fused residual-add + RMSNorm + quantisation op.
//
// Operation (vLLM docs "Fusion torch.compile passes", section "RMSNorm +
// Quantization (fuse_norm_quant)"; NVFP4 variant from the vLLM PR #51925
// summary, "Motivation"): per row, h = T(x + residual) written back as the
// updated residual, y = h * (1 / sqrt(mean(h^2) + eps)) * w, and y quantised
// to FP8 E4M3 (static / per-token / per-group scale) or NVFP4, all in one pass
// over HBM.
//
// Mapping: one CTA per row; thread t owns the J consecutive 16-byte chunks
// t*J .. t*J+J-1 (8 elements each) of x, residual and weight.  That mapping
// realises the canonical pairwise tree of the sum of squares without any
// reordering: the tree over 8 elements inside a chunk, then over the J chunks
// of a thread, then over lanes (xor butterfly), then over warps (one warp's
// butterfly over the 32 warp sums, zero-padded).  Zero padding is exact.
#pragma once

#include "rmsq_device.cuh"

namespace rmsq {

enum Mode : int {
    kFp8Static = 0,
    kFp8PerToken = 1,
    kFp8G128Row = 2,
    kFp8G128Col = 3,
    kFp8G64Row = 4,
    kFp8G64Col = 5,
    kNvfp4 = 6,
};

struct RowArgs {
    const uint4* x;
    const uint4* res;
    const uint4* w;
    uint4* res_out;
    uint8_t* q;
    void* scales;
    const float* scale_in;
    float eps;
    int n;        // rows
    int hidden;   // elements per row
    int chunks;   // hidden / 8
};

template <int MODE> struct ModeTraits {
    static constexpr int group = (MODE == kFp8G128Row || MODE == kFp8G128Col) ? 128
                               : (MODE == kFp8G64Row || MODE == kFp8G64Col) ? 64 : 0;
    static constexpr bool col = (MODE == kFp8G128Col || MODE == kFp8G64Col);
};

template <class E, int MODE, bool RES, int J>
__global__ void __launch_bounds__(1024) rows_kernel(const RowArgs a) {
    __shared__ float s_sum[32];
    __shared__ float s_max[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row = blockIdx.x;
    const int64_t base = (int64_t)row * a.chunks;

    // ---- loads: everything this thread needs, issued up front ----
    uint4 xv[J], rv[J], wv[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int c = tid * J + j;
        xv[j] = rv[j] = wv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (c < a.chunks) {
            xv[j] = ld_act(a.x + base + c);
            if constexpr (RES) rv[j] = ld_act(a.res + base + c);
            wv[j] = ld_weight(a.w + c);
        }
    }

    // ---- residual add (rounded to T), residual_out, sum of squares ----
    uint32_t hw[J][4];
    float part[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int c = tid * J + j;
        const uint32_t xs[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        if constexpr (RES) {
            const uint32_t rs[4] = {rv[j].x, rv[j].y, rv[j].z, rv[j].w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                hw[j][k] = E::pack(__fadd_rn(E::lo(xs[k]), E::lo(rs[k])),
                                   __fadd_rn(E::hi(xs[k]), E::hi(rs[k])));
            if (c < a.chunks)
                st_stream(a.res_out + base + c, make_uint4(hw[j][0], hw[j][1], hw[j][2], hw[j][3]));
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) hw[j][k] = xs[k];
        }
        float h[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) { h[2 * k] = E::lo(hw[j][k]); h[2 * k + 1] = E::hi(hw[j][k]); }
        part[j] = leaf8_sumsq(h);
    }
    float acc;
    if constexpr (J == 1) acc = part[0];
    else if constexpr (J == 2) acc = __fadd_rn(part[0], part[1]);
    else acc = __fadd_rn(__fadd_rn(part[0], part[1]), __fadd_rn(part[2], part[3]));
    static_assert(J == 1 || J == 2 || J == 4, "J must be 1, 2 or 4");

    acc = warp_tree_sum(acc);
    if (lane == 0) s_sum[warp] = acc;
    __syncthreads();
    const float total = warp_tree_sum(lane < nwarps ? s_sum[lane] : 0.0f);

    const float ms = __fdiv_rn(total, (float)a.hidden);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));

    // ---- y = (h * inv) * w in fp32 ----
    float y[J][8];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const uint32_t ws[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[j][2 * k] = __fmul_rn(__fmul_rn(E::lo(hw[j][k]), inv), E::lo(ws[k]));
            y[j][2 * k + 1] = __fmul_rn(__fmul_rn(E::hi(hw[j][k]), inv), E::hi(ws[k]));
        }
    }

    // ---- quantisation ----
    if constexpr (MODE == kNvfp4) {
        // 16-element blocks = chunk pairs (2m, 2m+1): a lane pair when J == 1,
        // inside the thread otherwise.
        const float gs = __ldg(a.scale_in);
        uint8_t* bsc = static_cast<uint8_t*>(a.scales) + (int64_t)row * (a.hidden / 16);
        uint32_t* qrow = reinterpret_cast<uint32_t*>(a.q + (int64_t)row * (a.hidden / 2));
#pragma unroll
        for (int j = 0; j < J; j += (J == 1 ? 1 : 2)) {
            float m = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(y[j][k]));
            if constexpr (J == 1) {
                m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(y[j + 1][k]));
            }
            const uint32_t sb = e4m3x2(__fmul_rn(__fdiv_rn(m, 6.0f), gs), 0.0f) & 0xffu;
            const float d = e4m3_value_nonneg(sb);
            const float r = (d == 0.0f) ? 0.0f : __fdiv_rn(gs, d);
            const int c = tid * J + j;
            const int nc = (J == 1) ? 1 : 2;
#pragma unroll
            for (int u = 0; u < nc; ++u) {
                float v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = __fmul_rn(y[j + u][k], r);
                if (c + u < a.chunks) st_stream(qrow + c + u, e2m1x8(v));
            }
            if (c < a.chunks && (c & 1) == 0) bsc[c >> 1] = (uint8_t)sb;
        }
    } else {
        float sval[J];
        if constexpr (MODE == kFp8Static) {
            const float s = __ldg(a.scale_in);
#pragma unroll
            for (int j = 0; j < J; ++j) sval[j] = s;
        } else if constexpr (MODE == kFp8PerToken) {
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j)
#pragma unroll
                for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(y[j][k]));
            m = lanes_max<32>(m);
            if (lane == 0) s_max[warp] = m;
            __syncthreads();
            m = lanes_max<32>(lane < nwarps ? s_max[lane] : 0.0f);
            const float s = fmaxf(__fdiv_rn(m, 448.0f), 1e-12f);
            if (tid == 0) static_cast<float*>(a.scales)[row] = s;
#pragma unroll
            for (int j = 0; j < J; ++j) sval[j] = s;
        } else {
            constexpr int G = ModeTraits<MODE>::group;
            constexpr int LANES = G / 8 / J;   // threads sharing one group
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j)
#pragma unroll
                for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(y[j][k]));
            m = lanes_max<LANES>(m);
            const float s = fmaxf(__fdiv_rn(m, 448.0f), 1e-12f);
            const int c0 = tid * J;
            if (c0 < a.chunks && (c0 % (G / 8)) == 0) {
                const int g = c0 / (G / 8);
                float* sc = static_cast<float*>(a.scales);
                if constexpr (ModeTraits<MODE>::col) sc[(int64_t)g * a.n + row] = s;
                else sc[(int64_t)row * (a.hidden / G) + g] = s;
            }
#pragma unroll
            for (int j = 0; j < J; ++j) sval[j] = s;
        }
        uint2* qrow = reinterpret_cast<uint2*>(a.q + (int64_t)row * a.hidden);
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int c = tid * J + j;
            const uint2 codes = fp8_chunk(y[j], sval[j]);
            if (c < a.chunks) st_stream(qrow + c, codes);
        }
    }
}

}  // namespace rmsq

// Per-row arithmetic shared by the row kernels of the fused residual-add +
// RMSNorm + quantisation op.
//
// Operation (vLLM docs "Fusion torch.compile passes", section "RMSNorm +
// Quantization (fuse_norm_quant)"; NVFP4 variant from the vLLM PR #51925
// summary, "Motivation"): per row, h = T(x + residual) written back as the
// updated residual, y = h * (1 / sqrt(mean(h^2) + eps)) * w, and y quantised
// to FP8 E4M3 (static / per-token / per-group scale) or NVFP4.
//
// Data-to-thread mapping used by every kernel: thread t owns the J
// consecutive 16-byte chunks t*J .. t*J+J-1 (8 elements each) of a row.  That
// realises the canonical pairwise tree of the sum of squares without any
// reordering: tree over the 8 elements of a chunk, over the J chunks of a
// thread, over lanes (xor butterfly), over warps (one warp's butterfly over
// the zero-padded warp sums).  Zero padding is exact.
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
    // First pass of NVFP4 with a data-derived global scale: residual add,
    // RMSNorm, the row's inv_rms stored in the workspace and the running
    // CTA's amax of y into its slot of the workspace; no codes.
    kNormAmax = 7,
    // The norm alone (the first op of the unfused sequence): y rounded to
    // the activation type, stored at q as a [n, hidden] T tensor.
    kNormOnly = 8,
};

// Workspace of the data-derived NVFP4 global scale: the fp32 inv_rms of row t
// sits at float index kWsInvOffset + t, and the amax of |y| over the rows of
// CTA b of the first pass at float index kWsInvOffset + n + b (at most one
// CTA per row, so n slots suffice).  The second pass takes the batch amax as
// the max of those partial maxima: nothing has to be zeroed before a call.
constexpr int kWsInvOffset = 64;

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
    float inv_hidden_pow2;   // 2^-k when hidden = 2^k, else 0
    // Chunk pairs (2m, 2m+1) of a row are stored (and, by the direct kernel,
    // loaded) as one access: set when `chunks` is even, x / residual /
    // residual_out start on 32 bytes and the codes on 16 bytes.
    bool pair;
    bool e8m0;        // dynamic scales rounded up to a power of two
    bool ue8m0;       // ... and stored as one UE8M0 byte each (the biased exponent)
    int col_stride;   // column-major scale stride: n, or n rounded up to 16 bytes
};

// The smallest power of two >= s for a positive normal s: s itself when its
// fraction bits are zero, else the next binade's first value (exact).
__device__ __forceinline__ float pow2_ceil(float s) {
    const uint32_t u = __float_as_uint(s);
    return (u & 0x007fffffu) == 0u ? s : __uint_as_float((u & 0x7f800000u) + 0x00800000u);
}

// A dynamic FP8 scale into element i of the scale tensor: fp32, or with the
// UE8M0 byte option its biased exponent (the scale is then a power of two,
// 2^(byte - 127)).
__device__ __forceinline__ void store_scale(const RowArgs& a, int64_t i, float s) {
    if (a.ue8m0) static_cast<uint8_t*>(a.scales)[i] = static_cast<uint8_t>(__float_as_uint(s) >> 23);
    else static_cast<float*>(a.scales)[i] = s;
}

template <int MODE> struct ModeTraits {
    static constexpr int group = (MODE == kFp8G128Row || MODE == kFp8G128Col) ? 128
                               : (MODE == kFp8G64Row || MODE == kFp8G64Col) ? 64 : 0;
    static constexpr bool col = (MODE == kFp8G128Col || MODE == kFp8G64Col);
    static constexpr bool needs_scale_in = (MODE == kFp8Static || MODE == kNvfp4);
};

// h = T(x + r) for the thread's chunks (h = x without a residual), the
// residual write-back, and the thread's partial of the sum-of-squares tree.
// Chunks at or beyond `chunks` hold zeros and are not stored.
// With `pair` (J >= 2, chunks even) each chunk pair of the write-back is one
// 32-byte store.  KEEP: the write-back is read again by a later phase, so it
// is stored at normal L2 priority instead of streamed.
template <class E, bool RES, int J, bool KEEP = false>
__device__ __forceinline__ float combine_chunks(const uint4 (&xv)[J], const uint4 (&rv)[J],
                                                uint32_t (&hw)[J][4], uint4* res_out_row,
                                                int c0, int chunks, bool pair) {
    float part[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        hw[j][0] = xv[j].x; hw[j][1] = xv[j].y; hw[j][2] = xv[j].z; hw[j][3] = xv[j].w;
        if constexpr (RES) {
            const uint32_t rs[4] = {rv[j].x, rv[j].y, rv[j].z, rv[j].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) hw[j][k] = E::add2(hw[j][k], rs[k]);
        }
    }
    if constexpr (RES) {
        if (J >= 2 && pair) {
#pragma unroll
            for (int j = 0; j + 1 < J; j += 2)
                if (c0 + j < chunks) {
                    if constexpr (KEEP) st_keep_pair(res_out_row + c0 + j, hw[j], hw[j + 1]);
                    else st_stream_pair(res_out_row + c0 + j, hw[j], hw[j + 1]);
                }
        } else {
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (c0 + j < chunks) {
                    const uint4 v = make_uint4(hw[j][0], hw[j][1], hw[j][2], hw[j][3]);
                    if constexpr (KEEP) st_keep(res_out_row + c0 + j, v);
                    else st_stream(res_out_row + c0 + j, v);
                }
        }
    }
    float h[J][8];
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) { h[j][2 * k] = E::lo(hw[j][k]); h[j][2 * k + 1] = E::hi(hw[j][k]); }
    if constexpr (J == 1) {
        part[0] = leaf8_sumsq(h[0]);
    } else {
#pragma unroll
        for (int j = 0; j < J; j += 2) {   // two chunks' leaf trees in packed pairs
            const float2 pp = leaf8_sumsq2(h[j], h[j + 1]);
            part[j] = pp.x;
            part[j + 1] = pp.y;
        }
    }
    static_assert(J == 1 || J == 2 || J == 4, "J must be 1, 2 or 4");
    if constexpr (J == 1) return part[0];
    else if constexpr (J == 2) return __fadd_rn(part[0], part[1]);
    else return __fadd_rn(__fadd_rn(part[0], part[1]), __fadd_rn(part[2], part[3]));
}

// 1 / sqrt(S / hidden + eps), each step correctly rounded.  For hidden = 2^k
// the division is the exact scaling S * 2^-k: the same real number, so the
// same correctly rounded result, without the divide.
__device__ __forceinline__ float inv_rms(float total, const RowArgs& a) {
    const float ms = a.inv_hidden_pow2 != 0.0f ? __fmul_rn(total, a.inv_hidden_pow2)
                                               : __fdiv_rn(total, (float)a.hidden);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
}

// The weight chunks widened to fp32 (once per kernel in the pipelined
// kernel, where every row of the CTA uses them).
template <class E, int J>
__device__ __forceinline__ void widen_weights(const uint4 (&wv)[J], float (&w)[J][8]) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const uint32_t ws[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) { w[j][2 * k] = E::lo(ws[k]); w[j][2 * k + 1] = E::hi(ws[k]); }
    }
}

// y = (h * inv) * w in fp32 for the thread's chunks, in packed pairs: element
// k of chunks j and j + 1 (J >= 2), elements k and k + 2 of the chunk (J == 1).
template <class E, int J>
__device__ __forceinline__ void compute_y(const uint32_t (&hw)[J][4], const float (&w)[J][8], float inv,
                                          float (&y)[J][8]) {
    float h[J][8];
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) { h[j][2 * k] = E::lo(hw[j][k]); h[j][2 * k + 1] = E::hi(hw[j][k]); }
    const float2 iv = make_float2(inv, inv);
    if constexpr (J == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int k = (q & 1) + 4 * (q >> 1);
            const float2 t = mul2_rn(mul2_rn(make_float2(h[0][k], h[0][k + 2]), iv),
                                     make_float2(w[0][k], w[0][k + 2]));
            y[0][k] = t.x; y[0][k + 2] = t.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < J; j += 2)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 t = mul2_rn(mul2_rn(make_float2(h[j][k], h[j + 1][k]), iv),
                                         make_float2(w[j][k], w[j + 1][k]));
                y[j][k] = t.x; y[j + 1][k] = t.y;
            }
    }
}

// E4M3 codes of y / s for the thread's chunks of `row`, stored.  DYN: s is a
// dynamic scale (within [1e-12, 2^120)), whose reciprocal takes the
// single-instruction form (fp8_recips_dyn).
template <int J, bool DYN = false>
__device__ __forceinline__ void store_fp8_codes(const RowArgs& a, int row, const float (&y)[J][8], float s,
                                                int c0) {
    const Fp8Recips rc = DYN ? fp8_recips_dyn(s) : fp8_recips(s);
    uint2* qrow = reinterpret_cast<uint2*>(a.q + (int64_t)row * a.hidden);
    uint2 codes[J];
    if constexpr (J == 1) {
        codes[0] = fp8_chunk(y[0], s, rc);
    } else {
#pragma unroll
        for (int j = 0; j < J; j += 2) fp8_chunk2(y[j], y[j + 1], s, rc, codes[j], codes[j + 1]);
    }
    if (J >= 2 && a.pair) {   // a chunk pair's 16 code bytes in one store
#pragma unroll
        for (int j = 0; j + 1 < J; j += 2)
            if (c0 + j < a.chunks)
                st_stream(reinterpret_cast<uint4*>(qrow + c0 + j),
                          make_uint4(codes[j].x, codes[j].y, codes[j + 1].x, codes[j + 1].y));
    } else {
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (c0 + j < a.chunks) st_stream(qrow + c0 + j, codes[j]);
    }
}

// FP8 per-token, before the CTA barrier: the warp's amax of |y| into s_max[warp].
template <int J>
__device__ __forceinline__ void per_token_warp_amax(const float (&y)[J][8], float* s_max, int lane, int warp) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < J; ++j)
        m = max_abs8(m, y[j]);
    m = warp_max_nonneg(m);
    if (lane == 0) s_max[warp] = m;
}

// FP8 per-token, after the barrier: s = max(amax / 448, 1e-12) from the warp
// slots, stored by thread 0, and the row's codes.
template <int J>
__device__ __forceinline__ void per_token_finish(const RowArgs& a, int row, const float (&y)[J][8],
                                                 const float* s_max, int tid, int nwarps) {
    const int lane = tid & 31;
    const float m = warp_max_nonneg(lane < nwarps ? s_max[lane] : 0.0f);
    float s = fmaxf(__fdiv_rn(m, 448.0f), 1e-12f);
    if (a.e8m0) s = pow2_ceil(s);
    if (tid == 0) store_scale(a, row, s);
    store_fp8_codes<J, true>(a, row, y, s, tid * J);
}

// The quantisation of `MODE` of the fp32 values y of the thread's chunks
// (chunks c0 .. c0+J-1 of `row`; c0 = tid*J unless the CTA covers a segment
// of the row) and all its stores.  `sin` is the static scale (FP8 static) or
// the global scale (NVFP4); `rtab` the NVFP4 table of gs / decode(code)
// (fill_nvfp4_rtab), else unused.  FP8 per-token does a CTA-wide amax through
// `s_max` (32 floats) and one __syncthreads, over the whole row (c0 = tid*J);
// every thread of the CTA must call this.
template <int MODE, int J>
__device__ __forceinline__ void quantize_y(const RowArgs& a, int row, const float (&y)[J][8], float sin,
                                           const float* rtab, float* s_max, int tid, int nwarps, int c0) {
    const int lane = tid & 31, warp = tid >> 5;
    if constexpr (MODE == kFp8PerToken) {
        per_token_warp_amax<J>(y, s_max, lane, warp);
        __syncthreads();
        per_token_finish<J>(a, row, y, s_max, tid, nwarps);
    } else if constexpr (MODE == kNvfp4) {
        // 16-element blocks = chunk pairs (2m, 2m+1): a lane pair when J == 1,
        // inside the thread otherwise.
        const float gs = sin;
        uint8_t* bsc = static_cast<uint8_t*>(a.scales) + (int64_t)row * (a.hidden / 16);
        uint32_t* qrow = reinterpret_cast<uint32_t*>(a.q + (int64_t)row * (a.hidden / 2));
#pragma unroll
        for (int j = 0; j < J; j += (J == 1 ? 1 : 2)) {
            float m = 0.0f;
            m = max_abs8(m, y[j]);
            if constexpr (J == 1) {
                m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
            } else {
                m = max_abs8(m, y[j + 1]);
            }
            const uint32_t sb = e4m3x2(__fmul_rn(__fdiv_rn(m, 6.0f), gs), 0.0f) & 0xffu;
            const float r = rtab[sb];      // gs / decode(sb), 0 for a zero block scale
            const int c = c0 + j;
            constexpr int NC = (J == 1) ? 1 : 2;
            uint32_t codes[NC];
            const float2 rr = make_float2(r, r);
            if constexpr (NC == 1) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int k = (q & 1) + 4 * (q >> 1);
                    const float2 t = mul2_rn(make_float2(y[j][k], y[j][k + 2]), rr);
                    v[k] = t.x; v[k + 2] = t.y;
                }
                codes[0] = e2m1x8(v);
            } else {
                float v0[8], v1[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 t = mul2_rn(make_float2(y[j][k], y[j + 1][k]), rr);
                    v0[k] = t.x; v1[k] = t.y;
                }
                codes[0] = e2m1x8(v0);
                codes[NC - 1] = e2m1x8(v1);
            }
            if (NC == 2 && a.pair) {   // the block's 8 code bytes in one store
                if (c < a.chunks) st_stream(reinterpret_cast<uint2*>(qrow + c), make_uint2(codes[0], codes[NC - 1]));
            } else {
#pragma unroll
                for (int u = 0; u < NC; ++u)
                    if (c + u < a.chunks) st_stream(qrow + c + u, codes[u]);
            }
            if (c < a.chunks && (c & 1) == 0) bsc[c >> 1] = (uint8_t)sb;
        }
    } else {
        float s;
        if constexpr (MODE == kFp8Static) {
            s = sin;
        } else {
            constexpr int G = ModeTraits<MODE>::group;
            constexpr int LANES = G / 8 / J;   // threads sharing one group
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j) m = max_abs8(m, y[j]);
            m = lanes_max<LANES>(m);
            s = fmaxf(__fdiv_rn(m, 448.0f), 1e-12f);
            if (a.e8m0) s = pow2_ceil(s);
            if (c0 < a.chunks && (c0 % (G / 8)) == 0) {
                const int g = c0 / (G / 8);
                if constexpr (ModeTraits<MODE>::col) store_scale(a, (int64_t)g * a.col_stride + row, s);
                else store_scale(a, (int64_t)row * (a.hidden / G) + g, s);
            }
        }
        store_fp8_codes<J, MODE != kFp8Static>(a, row, y, s, c0);
    }
}

// y = (h * inv) * w, then the quantisation of `MODE` (quantize_y), or for
// kNormAmax the row's inv_rms into the workspace and the running amax.
template <class E, int MODE, int J>
__device__ __forceinline__ void quantize_row(const RowArgs& a, int row, const uint32_t (&hw)[J][4],
                                             const float (&wv)[J][8], float inv, float sin,
                                             const float* rtab, float* s_max, int tid, int nwarps,
                                             float& run_max) {
    float y[J][8];
    compute_y<E, J>(hw, wv, inv, y);
    if constexpr (MODE == kNormAmax) {
#pragma unroll
        for (int j = 0; j < J; ++j) run_max = max_abs8(run_max, y[j]);
        if (tid == 0) static_cast<float*>(a.scales)[kWsInvOffset + row] = inv;
    } else if constexpr (MODE == kNormOnly) {
        (void)run_max;
        uint4* yrow = reinterpret_cast<uint4*>(a.q) + (int64_t)row * a.chunks;
        const int c0 = tid * J;
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (c0 + j < a.chunks)
                st_stream(yrow + c0 + j, make_uint4(E::pack(y[j][0], y[j][1]), E::pack(y[j][2], y[j][3]),
                                                    E::pack(y[j][4], y[j][5]), E::pack(y[j][6], y[j][7])));
    } else {
        (void)run_max;
        quantize_y<MODE, J>(a, row, y, sin, rtab, s_max, tid, nwarps, tid * J);
    }
}

// End of a kNormAmax launch: CTA-wide max of the threads' running amax into
// the CTA's slot of the workspace.  Every thread of the CTA calls it (two
// __syncthreads); `s_max` is 32 floats of shared memory.
__device__ __forceinline__ void flush_amax(const RowArgs& a, float run_max, float* s_max, int tid,
                                           int nwarps) {
    const int lane = tid & 31, warp = tid >> 5;
    const float m = warp_max_nonneg(run_max);
    __syncthreads();
    if (lane == 0) s_max[warp] = m;
    __syncthreads();
    if (tid == 0) {
        float t = 0.0f;
        for (int w = 0; w < nwarps; ++w) t = fmaxf(t, s_max[w]);
        static_cast<float*>(a.scales)[kWsInvOffset + a.n + blockIdx.x] = t;
    }
}

}  // namespace rmsq

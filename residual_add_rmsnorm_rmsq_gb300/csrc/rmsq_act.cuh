// SiLU+Mul + quantisation: the activation of a gated MLP fused with the
// quantisation of its result (vLLM docs "Fusion torch.compile passes",
// section "SiLU+Mul + Quantization (fuse_act_quant)": silu_and_mul on the
// gated up-projection and the following quantisation in one kernel, without
// the full-precision activation tensor in between).
//
// Each row of the input holds the gate g in its first d elements and the up
// projection u in the next d; a = silu(g) * u in fp32 with
// silu(g) = g / (1 + e^-g), then exactly the quantisation epilogue of the
// norm kernels (quantize_y) on a.  One CTA per row, thread t on the chunks
// t*J .. t*J+J-1 of the row, as in the direct norm kernel.
//
// silu(g) is g times the approximate reciprocal of 1 + e^-g (the result is
// compared with the oracle's correctly rounded silu within a bound derived
// from these steps).  e^x is evaluated with W. J. Cody and W. Waite's
// argument reduction ("Software Manual for the Elementary Functions", 1980):
// x = n ln2 + r with n = rint(x log2 e) and ln2 split in a high part of 15
// significant bits (n ln2_hi is exact) and the rest, r formed by two fused
// multiply-adds; e^r = 2^(r log2 e) by the hardware approximation of 2^x on
// that small argument; then the scaling by 2^n in two power-of-two factors
// (the second is 1 unless 2^n is not a normal binary32).  Within about 2.4
// ulp of e^x; every step is deterministic, done in packed pairs where two
// elements take the same step.
#pragma once

#include "rmsq_dispatch.cuh"

namespace rmsq {

__device__ __forceinline__ float pow2_bits(int k) { return __int_as_float((k + 127) << 23); }

// 2^a by the hardware approximation (ex2.approx, about two ulps).
__device__ __forceinline__ float ex2_approx(float a) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// The same approximation without the handling of subnormal inputs and
// results (a single hardware instruction): identical to ex2_approx for every
// |a| <= 0.5 (checked exhaustively on GB300), where 2^a is normal and a
// subnormal a gives 1 either way.
__device__ __forceinline__ float ex2_approx_ftz(float a) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

// rint(t) and 2^rint(t) for |t| < 2^22 without a float-to-integer conversion:
// t + 1.5 * 2^23 lands in [2^23, 2^24), where the spacing of binary32 is 1, so
// the addition rounds t to the nearest integer (ties to even, as rint), whose
// value minus 1.5 * 2^23 is n and whose bit pattern is 0x4b400000 + n.
constexpr float kRintMagic = 12582912.0f;   // 1.5 * 2^23
__device__ __forceinline__ int rint_bits_to_int(float tm) { return __float_as_int(tm) - 0x4b400000; }

// e^x for two elements.
__device__ __forceinline__ float2 exp_cw2(float2 x) {
    const float hi_lim = 89.0f, lo_lim = -104.0f;    // e^89 > FLT_MAX; e^-104 < half the least subnormal
    const float2 xc = make_float2(fminf(fmaxf(x.x, lo_lim), hi_lim), fminf(fmaxf(x.y, lo_lim), hi_lim));
    const float log2e = 1.44269502162933349609375f;  // RN(log2 e)
    const float ln2_hi = 0.693145751953125f;         // 0x3f317200
    const float ln2_lo = 1.428606765330187045e-06f;  // RN(ln2 - ln2_hi)
    const float2 t = mul2_rn(xc, make_float2(log2e, log2e));
    const float2 tm = add2_rn(t, make_float2(kRintMagic, kRintMagic));   // |t| < 151
    const float2 n = add2_rn(tm, make_float2(-kRintMagic, -kRintMagic));  // rint(t)
    const float2 nn = make_float2(-n.x, -n.y);
    const float2 r = fma2_rn(nn, make_float2(ln2_lo, ln2_lo), fma2_rn(nn, make_float2(ln2_hi, ln2_hi), xc));
    const float2 rl = mul2_rn(r, make_float2(log2e, log2e));
    const float2 p = make_float2(ex2_approx(rl.x), ex2_approx(rl.y));
    // 2^k = 2^ka * 2^kb with both factors normal: ka = min(k, 127), or k + 64
    // below -126; kb = k - ka (0 unless 2^k alone is out of the normal range).
    const int k0 = rint_bits_to_int(tm.x), k1 = rint_bits_to_int(tm.y);
    const int a0 = k0 < -126 ? k0 + 64 : min(k0, 127), a1 = k1 < -126 ? k1 + 64 : min(k1, 127);
    float2 e = mul2_rn(mul2_rn(p, make_float2(pow2_bits(a0), pow2_bits(a1))),
                       make_float2(pow2_bits(k0 - a0), pow2_bits(k1 - a1)));
    const float inf = __int_as_float(0x7f800000);
    e.x = x.x != x.x ? x.x : x.x > hi_lim ? inf : x.x < lo_lim ? 0.0f : e.x;
    e.y = x.y != x.y ? x.y : x.y > hi_lim ? inf : x.y < lo_lim ? 0.0f : e.y;
    return e;
}

// e^x for two elements with |x| <= 87: the same steps as exp_cw2, where
// nothing is clamped, 2^n is a normal binary32 (|n| <= 126) and no special
// value arises, so the result is identical with a single scaling factor; the
// reduced argument is within 0.5 + 2^-16 in magnitude, so the plain hardware
// 2^x gives the same value as ex2_approx.
__device__ __forceinline__ float2 exp_cw2_mid(float2 x) {
    const float log2e = 1.44269502162933349609375f, ln2_hi = 0.693145751953125f, ln2_lo = 1.428606765330187045e-06f;
    const float2 t = mul2_rn(x, make_float2(log2e, log2e));
    const float2 tm = add2_rn(t, make_float2(kRintMagic, kRintMagic));
    const float2 n = add2_rn(tm, make_float2(-kRintMagic, -kRintMagic));
    const float2 nn = make_float2(-n.x, -n.y);
    const float2 r = fma2_rn(nn, make_float2(ln2_lo, ln2_lo), fma2_rn(nn, make_float2(ln2_hi, ln2_hi), x));
    const float2 rl = mul2_rn(r, make_float2(log2e, log2e));
    const float2 p = make_float2(ex2_approx_ftz(rl.x), ex2_approx_ftz(rl.y));
    return mul2_rn(p, make_float2(pow2_bits(rint_bits_to_int(tm.x)), pow2_bits(rint_bits_to_int(tm.y))));
}

// 1 / x by the hardware approximation: within one ulp over the whole range
// (subnormal results kept).
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// The same without the handling of subnormal inputs and results (a single
// hardware instruction): identical to rcp_approx for every x in [1, 2^126)
// (checked exhaustively on GB300), which holds 1 + e^-g for |g| <= 87.
__device__ __forceinline__ float rcp_approx_ftz(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// a = silu(g) * u = g * (1 / (1 + e^-g)) * u for two elements; MID: both
// |g| <= 87 (e^-g by exp_cw2_mid, else by exp_cw2).  The quotient is g times
// the approximate reciprocal of 1 + e^-g (one ulp), so silu is within
// 8.8 * 2^-24 of its exact value: e^-g 2.4 ulp, the sum, the reciprocal and
// the product.
template <bool MID = false>
__device__ __forceinline__ float2 silu_mul2(float2 g, float2 u) {
    const float2 e = MID ? exp_cw2_mid(make_float2(-g.x, -g.y)) : exp_cw2(make_float2(-g.x, -g.y));
    const float2 den = add2_rn(make_float2(1.0f, 1.0f), e);
    const float2 s = MID ? mul2_rn(g, make_float2(rcp_approx_ftz(den.x), rcp_approx_ftz(den.y)))
                         : mul2_rn(g, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
    return mul2_rn(s, u);
}

// a for the thread's J chunks of gate and up.
template <class E, int J, bool MID>
__device__ __forceinline__ void act_chunks(const uint4 (&gv)[J], const uint4 (&uv)[J], float (&y)[J][8]) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const uint32_t g[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
        const uint32_t u[4] = {uv[j].x, uv[j].y, uv[j].z, uv[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 v = silu_mul2<MID>(make_float2(E::lo(g[k]), E::hi(g[k])), make_float2(E::lo(u[k]), E::hi(u[k])));
            y[j][2 * k] = v.x;
            y[j][2 * k + 1] = v.y;
        }
    }
}

// Threads per CTA of the activation kernel.  A CTA covers a segment of
// `seg` chunks of one row (the whole row for FP8 per-token, whose scale needs
// the row's amax), thread t the chunks base + t*J .. base + t*J+J-1.
constexpr int kActMaxThreads = 512;

// SILU: the input row is gate | up and y = silu(gate) * up; otherwise the
// input is a [n, hidden] T tensor quantised as it is (the second op of the
// unfused sequence).
template <class E, int MODE, int J, bool SILU>
__device__ __forceinline__ void act_rows_body(const RowArgs& a, const int segs, const int seg) {
    __shared__ float s_max[32];
    __shared__ float s_rtab[MODE == kNvfp4 ? 128 : 1];
    const int tid = threadIdx.x, nwarps = blockDim.x >> 5;
    const int row = blockIdx.x / segs;
    const int c0 = (blockIdx.x - row * segs) * seg + tid * J;
    allow_dependents();
    grid_dependency_wait();

    // a.x: the [n, 2d] input (gate chunks of the row, then up chunks), or
    // the [n, d] input without SILU (read as the "gate" half)
    const uint4* gp = a.x + (int64_t)row * (SILU ? 2 : 1) * a.chunks;
    const uint4* up = gp + a.chunks;
    uint4 gv[J], uv[J];
#pragma unroll
    for (int j = 0; j < J; ++j) gv[j] = uv[j] = make_uint4(0u, 0u, 0u, 0u);
    if (J >= 2 && a.pair) {   // chunks even: a chunk pair is in the row or wholly past it
#pragma unroll
        for (int j = 0; j + 1 < J; j += 2)
            if (c0 + j < a.chunks) {
                ld_act_pair(gp + c0 + j, gv[j], gv[j + 1]);
                if constexpr (SILU) ld_act_pair(up + c0 + j, uv[j], uv[j + 1]);
            }
    } else {
#pragma unroll
        for (int j = 0; j < J; ++j)
            if (c0 + j < a.chunks) {
                gv[j] = ld_act(gp + c0 + j);
                if constexpr (SILU) uv[j] = ld_act(up + c0 + j);
            }
    }
    const float sin = ModeTraits<MODE>::needs_scale_in ? __ldg(a.scale_in) : 0.0f;
    if constexpr (MODE == kNvfp4) {
        fill_nvfp4_rtab(s_rtab, sin);
        __syncthreads();
    }

    float y[J][8];
    if constexpr (SILU) {
        // The usual case (every gate of the thread within +-87, tested on the
        // bit patterns: a NaN or infinity fails it) takes the shorter e^x
        // steps (the hardware 2^x on the reduced argument).
        uint32_t in_range = 0xffffffffu;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const uint32_t g[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) in_range &= __vcmpleu2(g[k] & 0x7fff7fffu, E::kBits87 * 0x10001u);
        }
        if (in_range == 0xffffffffu)
            act_chunks<E, J, true>(gv, uv, y);
        else
            act_chunks<E, J, false>(gv, uv, y);
    } else {
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const uint32_t g[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) { y[j][2 * k] = E::lo(g[k]); y[j][2 * k + 1] = E::hi(g[k]); }
        }
    }
    quantize_y<MODE, J>(a, row, y, sin, s_rtab, s_max, tid, nwarps, c0);
}

template <class E, int MODE, int J, bool SILU>
__global__ void __launch_bounds__(kActMaxThreads) act_rows_kernel(const RowArgs a, const int segs, const int seg) {
    act_rows_body<E, MODE, J, SILU>(a, segs, seg);
}

// The FP8 modes at four chunks per thread (the segment kernel) with their
// registers capped (compile-time tuning, results do not depend on it): 48
// lets 21 instead of 16 64-thread CTAs share an SM (Llama-8B MLP, 4096 x
// 14336: static 48.9 -> 46.1 us, group 128 50.3 -> 49.3 us); NVFP4 was 3 %
// slower under the cap and keeps the plain kernel.
#ifndef RMSQ_ACT_MAXNREG_FP8_J4
#define RMSQ_ACT_MAXNREG_FP8_J4 48
#endif
template <class E, int MODE, bool SILU>
__global__ void __maxnreg__(RMSQ_ACT_MAXNREG_FP8_J4)
act_rows_kernel_j4(const RowArgs a, const int segs, const int seg) {
    act_rows_body<E, MODE, 4, SILU>(a, segs, seg);
}

template <class E, int MODE, bool SILU>
const void* pick_act_j(int J) {
    switch (J) {
    case 1: return reinterpret_cast<const void*>(&act_rows_kernel<E, MODE, 1, SILU>);
    case 2: return reinterpret_cast<const void*>(&act_rows_kernel<E, MODE, 2, SILU>);
    case 4:
        if constexpr (MODE != kNvfp4) return reinterpret_cast<const void*>(&act_rows_kernel_j4<E, MODE, SILU>);
        else return reinterpret_cast<const void*>(&act_rows_kernel<E, MODE, 4, SILU>);
    default: return reinterpret_cast<const void*>(&act_rows_kernel<E, MODE, 8, SILU>);
    }
}

template <class E, bool SILU>
const void* pick_act(int mode, int J) {
    switch (mode) {
    case kFp8Static: return pick_act_j<E, kFp8Static, SILU>(J);
    case kFp8PerToken: return pick_act_j<E, kFp8PerToken, SILU>(J);
    case kFp8G128Row: return pick_act_j<E, kFp8G128Row, SILU>(J);
    case kFp8G128Col: return pick_act_j<E, kFp8G128Col, SILU>(J);
    case kFp8G64Row: return pick_act_j<E, kFp8G64Row, SILU>(J);
    case kFp8G64Col: return pick_act_j<E, kFp8G64Col, SILU>(J);
    case kNvfp4: return pick_act_j<E, kNvfp4, SILU>(J);
    default: return nullptr;
    }
}

// Segment shape for the modes without a row-wide scale (compile-time tuning;
// results do not depend on it): kActSegThreads threads of kActSegJ chunks.
// Small segments (many small CTAs per SM) hide the load latency of this
// arithmetic-heavy kernel best (measured on GB300: 64 x 4 beat 128 x 2,
// 256 x 2, 128 x 1 and 256 x 4 on 4096 x 14336).
#ifndef RMSQ_ACT_SEG_THREADS
#define RMSQ_ACT_SEG_THREADS 64
#endif
#ifndef RMSQ_ACT_SEG_J
#define RMSQ_ACT_SEG_J 4
#endif
constexpr int kActSegThreads = RMSQ_ACT_SEG_THREADS;
constexpr int kActSegJ = RMSQ_ACT_SEG_J;
static_assert(kActSegThreads * kActSegJ % 16 == 0, "segments hold whole groups of 128");

// One launch: la.x = gate_up [n, 2d] (silu) or the [n, d] tensor to
// quantise, la.hidden = d.
template <class E>
cudaError_t launch_act(const LaunchArgs& la, bool silu, cudaStream_t stream) {
    RowArgs a;
    a.x = static_cast<const uint4*>(la.x);
    a.res = nullptr;
    a.w = nullptr;
    a.res_out = nullptr;
    a.q = static_cast<uint8_t*>(la.q);
    a.scales = la.scales;
    a.scale_in = la.scale_in;
    a.eps = 0.0f;
    a.n = la.n;
    a.hidden = la.hidden;
    a.chunks = la.hidden / 8;
    a.inv_hidden_pow2 = 0.0f;
    a.pair = a.chunks % 2 == 0 && reinterpret_cast<uintptr_t>(la.x) % 32 == 0 &&
             reinterpret_cast<uintptr_t>(la.q) % 16 == 0;
    a.e8m0 = la.e8m0;
    a.ue8m0 = la.ue8m0;
    a.col_stride = la.col_stride;
    int J, threads, seg;
    if (la.mode == kFp8PerToken) {   // one CTA per row
        J = a.chunks <= 512 ? 1 : a.chunks <= 1024 ? 2 : a.chunks <= 2048 ? 4 : 8;
        threads = ((a.chunks + J - 1) / J + 31) / 32 * 32;
        seg = a.chunks;
    } else {
        // Equal segments of at most kActSegThreads * kActSegJ chunks, a
        // multiple of 16 chunks each (so that no group of 128 and no NVFP4
        // block straddles two).
        J = kActSegJ;
        const int most = kActSegThreads * kActSegJ;
        const int count = (a.chunks + most - 1) / most;
        seg = ((a.chunks + count - 1) / count + 15) / 16 * 16;
        threads = ((seg + J - 1) / J + 31) / 32 * 32;
    }
    const int segs = (a.chunks + seg - 1) / seg;
    const void* fn = silu ? pick_act<E, true>(la.mode, J) : pick_act<E, false>(la.mode, J);
    if (!fn) return cudaErrorInvalidValue;
    int segs_arg = segs, seg_arg = seg;
    void* params[] = {&a, &segs_arg, &seg_arg};
    return launch_kernel(fn, dim3((unsigned)((int64_t)a.n * segs)), dim3(threads), params, 0, stream);
}

}  // namespace rmsq

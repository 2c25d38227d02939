// Device helpers for the fused residual-add + RMSNorm + quantisation kernels (sm_103a).
//
// Number formats: OCP FP8 E4M3FN and FP4 E2M1, converted with the hardware
// cvt instructions (round to nearest even, .satfinite).  Every fp32 step uses
// the explicitly rounded intrinsics (__fadd_rn, __fmul_rn, __fdiv_rn,
// __fsqrt_rn) so that no multiply-add contraction changes a rounding.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rmsq {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Activation types: unpack one 32-bit word (two elements, the lower-addressed
// element in bits 0..15) to fp32, and pack two fp32 with round-to-nearest-even.
// ---------------------------------------------------------------------------
// add2: element-wise sum of two packed pairs, rounded once to nearest even.
// That equals rounding the fp32 sum to T: two values of T (8 / 11 significant
// bits) add exactly in fp32 unless their exponents are more than 15 / 13
// apart, and then the smaller one is below half an ulp of T, so neither
// rounding path can land on a tie of T and both give the larger operand.
struct Bf16T {
    static constexpr uint32_t kBits87 = 0x42aeu;    // 87.0 (magnitudes order like their bit patterns)
    static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
    static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    static __device__ __forceinline__ uint32_t add2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
};

struct Fp16T {
    static constexpr uint32_t kBits87 = 0x5570u;    // 87.0
    static __device__ __forceinline__ float lo(uint32_t w) {
        float f;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(w));
        return f;
    }
    static __device__ __forceinline__ float hi(uint32_t w) {
        float f;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(w));
        return f;
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    static __device__ __forceinline__ uint32_t add2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
};

// ---------------------------------------------------------------------------
// Global memory access.  Activations are touched once: no L1 allocation on
// loads, streaming (evict-first) stores.  The weight row is shared by every
// row of the launch and goes through the read-only path.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_act(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_weight(const uint4* p) {
    uint4 v;
    asm("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Two adjacent 16-byte chunks as one 256-bit access (sm_100 and later): a
// warp whose threads own chunk pairs then touches whole 32-byte sectors per
// instruction instead of half a sector per thread.  p must be 32-byte aligned.
__device__ __forceinline__ void ld_act_pair(const uint4* p, uint4& a, uint4& b) {
    asm volatile("ld.global.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
}

__device__ __forceinline__ void st_stream_pair(uint4* p, const uint32_t (&a)[4], const uint32_t (&b)[4]) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]),
                    "r"(b[3])
                 : "memory");
}

// Stores of data that is read again shortly (by a later phase of the same
// operation): plain write-back, the line stays in L2 at normal priority.
__device__ __forceinline__ void st_keep(uint4* p, uint4 v) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st_keep_pair(uint4* p, const uint32_t (&a)[4], const uint32_t (&b)[4]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "r"(b[2]),
                    "r"(b[3])
                 : "memory");
}

__device__ __forceinline__ void st_stream(uint2* p, uint2 v) {
    asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_stream(uint32_t* p, uint32_t v) {
    asm volatile("st.global.cs.b32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the kernel before it in the stream is still
// running.  grid_dependency_wait() returns once that kernel has completed and
// its memory operations are visible; every global memory access of a kernel
// comes after it.  (Launched without the attribute, it returns at once.)
// allow_dependents() lets the next kernel of the stream start early; that
// kernel in turn waits for this one to complete before touching memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Packed fp32 pairs (sm_100 and later): one instruction does two independent
// IEEE operations, each rounded to nearest-even exactly as the scalar .rn
// form (subnormals kept).  Without RMSQ_F32X2 the same pairs are done as two
// scalar operations, with identical results.
// ---------------------------------------------------------------------------
#ifndef RMSQ_F32X2
#define RMSQ_F32X2 1
#endif

__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
#if RMSQ_F32X2
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
#else
    return make_float2(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y));
#endif
}

__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
#if RMSQ_F32X2
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
#else
    return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
#endif
}

// a * b + c with one rounding (fused multiply-add) for two elements.  ptxas
// may also fuse a packed multiply feeding a packed add on its own (it did so
// for the Horner steps of an e^x evaluation), so every place whose result
// would change under such fusion states the fused form explicitly; the
// packed multiply-adds left elsewhere multiply exact squares or scale by
// powers of two, where fused and separate roundings agree.
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
#if RMSQ_F32X2
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
#else
    return make_float2(__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y));
#endif
}

// ---------------------------------------------------------------------------
// Conversions.
// ---------------------------------------------------------------------------

// Two fp32 -> two E4M3 codes: code(lo) in bits 0..7, code(hi) in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Eight fp32 -> eight E2M1 codes packed in one word: element k in nibble k.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Exact value of a non-negative, finite E4M3 code (the NVFP4 block scale):
// exponent field e, fraction m: e == 0 -> m * 2^-9, else (1 + m/8) * 2^(e-7).
__device__ __forceinline__ float e4m3_value_nonneg(uint32_t c) {
    const uint32_t e = (c >> 3) & 0xfu, m = c & 7u;
    return e == 0 ? __fmul_rn(__uint2float_rn(m), 0.001953125f)
                  : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// r = gs / decode(code) for every finite non-negative E4M3 code (0 for the
// zero code; 0x7f is NaN and never produced), in shared memory, so that the
// NVFP4 per-block division by the decoded block scale becomes a lookup.
// Filled cooperatively by the CTA; a barrier must follow before use.
__device__ __forceinline__ void fill_nvfp4_rtab(float* tab, float gs) {
    for (int c = threadIdx.x; c < 128; c += blockDim.x)
        tab[c] = (c == 0 || c == 127) ? 0.0f : __fdiv_rn(gs, e4m3_value_nonneg((uint32_t)c));
}

// E4M3 codes of y/s where the quotient is the correctly rounded fp32
// division, without a division per element: multiply by two bracketing
// reciprocals rdn = RN(RN(1/s) * (1 - 2^-20)) and rup = RN(RN(1/s) * (1 + 2^-20)).
// The products lie strictly below / above the rounded quotient in magnitude
// (the three roundings involved move a value by less than 3 * 2^-24
// relative), and the saturating nearest-even E4M3 cast is monotone, so equal
// codes at both ends are the code of the quotient.  Otherwise (about one
// element in 2^16) the quotient is computed with __fdiv_rn.

// Bracketing reciprocals of a scale s.  The argument above holds for any
// approximation of 1/s with relative error below 2^-18.1 once the bracket is
// widened to 1 -+ 2^-18, so the hardware's approximate reciprocal (documented
// error about one ulp, 2^-23) serves; a wider bracket only makes the exact
// fallback a little more frequent (about one chunk of eight in a thousand).
struct Fp8Recips {
    float rdn, rup;
};
__device__ __forceinline__ Fp8Recips fp8_recips(float s) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
    return {__fmul_rn(r, 0.999996185302734375f),       // 1 - 2^-18
            __fmul_rn(r, 1.000003814697265625f)};      // 1 + 2^-18
}

// The same for a dynamic scale (amax / 448, at least 1e-12, at most
// FLT_MAX / 448 < 2^120), with the single-instruction reciprocal that flushes
// subnormal inputs and results: for every s in [2^-126, 2^126) it equals the
// one above (checked exhaustively on GB300), and both s and 1 / s are normal
// there.  A static scale is the caller's and may lie outside that range.
__device__ __forceinline__ Fp8Recips fp8_recips_dyn(float s) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
    return {__fmul_rn(r, 0.999996185302734375f),       // 1 - 2^-18
            __fmul_rn(r, 1.000003814697265625f)};      // 1 + 2^-18
}

// E4M3 codes of v[k] / s, element k in byte k, for the eight elements of a
// chunk.  The bracketing test is applied to the whole chunk at once (one
// branch per eight elements); the rare chunk with a code that differs between
// the two ends is redone with correctly rounded divisions.
__device__ __forceinline__ uint2 fp8_chunk_exact(const float (&v)[8], float s) {
    uint32_t ex[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) ex[p] = e4m3x2(__fdiv_rn(v[2 * p], s), __fdiv_rn(v[2 * p + 1], s));
    return make_uint2(ex[0] | (ex[1] << 16), ex[2] | (ex[3] << 16));
}

// One chunk; the bracket products are formed in packed pairs (k, k + 1) and
// turned into codes right away.
__device__ __forceinline__ uint2 fp8_chunk(const float (&v)[8], float s, Fp8Recips rc) {
    uint32_t dn[4], up[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 e = make_float2(v[2 * p], v[2 * p + 1]);
        const float2 d = mul2_rn(e, make_float2(rc.rdn, rc.rdn));
        const float2 u = mul2_rn(e, make_float2(rc.rup, rc.rup));
        dn[p] = e4m3x2(d.x, d.y);
        up[p] = e4m3x2(u.x, u.y);
    }
    uint2 out = make_uint2(dn[0] | (dn[1] << 16), dn[2] | (dn[3] << 16));
    if (((out.x ^ (up[0] | (up[1] << 16))) | (out.y ^ (up[2] | (up[3] << 16)))) != 0u)
        out = fp8_chunk_exact(v, s);
    return out;
}

// Two chunks a, b under their own scales sa, sb (reciprocal brackets ra, rb):
// the bracket products are formed in packed pairs (a[k] * ra, b[k] * rb) and
// turned into codes right away; the codes of each bracket end are packed four
// to a word (byte permutes) and the two ends compared word by word.
__device__ __forceinline__ void fp8_chunk2s(const float (&a)[8], const float (&b)[8], float sa, float sb,
                                            Fp8Recips ra, Fp8Recips rb, uint2& ca, uint2& cb) {
    uint32_t da[4], db[4], ua[4], ub[4];
    const float2 dn = make_float2(ra.rdn, rb.rdn), up = make_float2(ra.rup, rb.rup);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 e0 = make_float2(a[2 * p], b[2 * p]), e1 = make_float2(a[2 * p + 1], b[2 * p + 1]);
        const float2 d0 = mul2_rn(e0, dn), d1 = mul2_rn(e1, dn);
        const float2 u0 = mul2_rn(e0, up), u1 = mul2_rn(e1, up);
        da[p] = e4m3x2(d0.x, d1.x);
        db[p] = e4m3x2(d0.y, d1.y);
        ua[p] = e4m3x2(u0.x, u1.x);
        ub[p] = e4m3x2(u0.y, u1.y);
    }
    ca = make_uint2(__byte_perm(da[0], da[1], 0x5410), __byte_perm(da[2], da[3], 0x5410));
    cb = make_uint2(__byte_perm(db[0], db[1], 0x5410), __byte_perm(db[2], db[3], 0x5410));
    const uint32_t diff = (ca.x ^ __byte_perm(ua[0], ua[1], 0x5410)) | (ca.y ^ __byte_perm(ua[2], ua[3], 0x5410)) |
                          (cb.x ^ __byte_perm(ub[0], ub[1], 0x5410)) | (cb.y ^ __byte_perm(ub[2], ub[3], 0x5410));
    if (diff != 0u) {   // rare: redo both chunks exactly
        ca = fp8_chunk_exact(a, sa);
        cb = fp8_chunk_exact(b, sb);
    }
}

// Two chunks a, b under one scale.
__device__ __forceinline__ void fp8_chunk2(const float (&a)[8], const float (&b)[8], float s, Fp8Recips rc,
                                           uint2& ca, uint2& cb) {
    fp8_chunk2s(a, b, s, s, rc, rc, ca, cb);
}

// Pairwise tree over the squares of eight consecutive elements, in packed
// pairs: (h0, h2) and (h1, h3) squared and added give the two level-1 nodes
// h0^2 + h1^2 and h2^2 + h3^2 at once (likewise for h4..h7).
__device__ __forceinline__ float leaf8_sumsq(const float (&h)[8]) {
    const float2 p02 = make_float2(h[0], h[2]), p13 = make_float2(h[1], h[3]);
    const float2 p46 = make_float2(h[4], h[6]), p57 = make_float2(h[5], h[7]);
    const float2 ab = add2_rn(mul2_rn(p02, p02), mul2_rn(p13, p13));
    const float2 cd = add2_rn(mul2_rn(p46, p46), mul2_rn(p57, p57));
    return __fadd_rn(__fadd_rn(ab.x, ab.y), __fadd_rn(cd.x, cd.y));
}

// The leaf trees of two chunks a, b at once, element k of both in one packed
// pair: returns (tree(a), tree(b)).
__device__ __forceinline__ float2 leaf8_sumsq2(const float (&a)[8], const float (&b)[8]) {
    float2 sq[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 p = make_float2(a[k], b[k]);
        sq[k] = mul2_rn(p, p);
    }
    const float2 l0 = add2_rn(sq[0], sq[1]), l1 = add2_rn(sq[2], sq[3]);
    const float2 l2 = add2_rn(sq[4], sq[5]), l3 = add2_rn(sq[6], sq[7]);
    return add2_rn(add2_rn(l0, l1), add2_rn(l2, l3));
}

// Butterfly sum over the 32 lanes: at step k lanes differing in bit k add
// their values, which is the pairwise tree over lane index (fp32 addition is
// commutative, so both partners hold the same node value).
__device__ __forceinline__ float warp_tree_sum(float v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Max over the 32 lanes of non-negative values: their bit patterns order like
// the values, so one integer max reduction does it.
__device__ __forceinline__ float warp_max_nonneg(float v) {
    return __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(v)));
}

// Pairwise tree over 16 / 32 consecutive floats of shared memory (16-byte
// aligned), read with 128-bit loads: the top levels of the canonical tree
// over warp sums, zero-padded.
template <int N>
__device__ __forceinline__ float smem_tree_sum(const float* p) {
    static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 slots");
    float v[N];
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float4 f = reinterpret_cast<const float4*>(p)[i];
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
#pragma unroll
    for (int len = N; len > 1; len >>= 1)
#pragma unroll
        for (int k = 0; k < len / 2; ++k) v[k] = __fadd_rn(v[2 * k], v[2 * k + 1]);
    return v[0];
}

// The same tree over the slots of `nwarps` warps (slots up to the next of
// 8 / 16 / MAX hold zeros): a zero-padded subtree adds only exact zeros, so
// summing the smallest power-of-two prefix that holds every warp's slot gives
// the full tree's value.
template <int MAX>
__device__ __forceinline__ float warp_slots_tree_sum(const float* p, int nwarps) {
    if (nwarps <= 8) return smem_tree_sum<8>(p);
    if constexpr (MAX >= 16) {
        if (MAX == 16 || nwarps <= 16) return smem_tree_sum<16>(p);
    }
    if constexpr (MAX >= 32) return smem_tree_sum<32>(p);
    return smem_tree_sum<MAX>(p);
}

// max(m, |a|, |b|) in one instruction; m >= 0.
__device__ __forceinline__ float max_abs3(float m, float a, float b) {
    float r;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(m), "f"(a), "f"(b));
    return r;
}

// max(m, |v_0|, ..., |v_7|), m >= 0.
__device__ __forceinline__ float max_abs8(float m, const float (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 8; k += 2) m = max_abs3(m, v[k], v[k + 1]);
    return m;
}

template <int LANES>
__device__ __forceinline__ float lanes_max(float v) {
#pragma unroll
    for (int o = 1; o < LANES; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (TMA, 1-D) into shared memory with mbarrier
// completion.  Addresses are 16-byte aligned and sizes multiples of 16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the other threads and to the
// asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Global -> shared bulk copy, completion counted on `bar` (transaction bytes).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` to complete; gives up (returns false) after
// kWaitLimitNs of wall time or 2^24 polls, whichever comes first.
constexpr uint64_t kWaitLimitNs = 100ull * 1000 * 1000;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

}  // namespace rmsq

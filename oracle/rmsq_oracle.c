/*
 * CPU oracle for the fused residual-add + RMSNorm + activation quantisation op.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the op computes.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference leg load it.  It shares no code, header,
 * table or constant with the CUDA library, and the CUDA library never calls it.
 *
 * What it follows:
 *  - vLLM docs, "Fusion torch.compile passes", section "RMSNorm + Quantization
 *    (fuse_norm_quant)": rms_norm(x) -> quant_fp8(y) and
 *    fused_add_rms_norm(x, residual) -> quant_fp8(y), the residual updated in
 *    place; schemes FP8 static per-tensor, FP8 dynamic per-token, FP8 dynamic
 *    per-token-group (128/64).
 *  - blog "[vLLM] Compilation Fusion Passes", sections "RMSNormQuantFusionPass"
 *    (eps 1e-5 / 1e-6), "Pattern matching structure" (result/input/weight/scale/
 *    epsilon), "Fused Add + RMSNorm + Group Quantization" (the FUSED_OPS keys:
 *    static tensor, dynamic token, dynamic 128-group, symmetric), "Why this
 *    design" (column-major scales).
 *  - vLLM PR #51925 summary (prhub), "Motivation" and "Key source snippets":
 *    residual update + RMSNorm, then block scales and conversion to FP4 with an
 *    fp32 activation (global) scale passed in.
 * The pages print no formula; the scale rules (amax/448 floored at 1e-12,
 * block scale e4m3(amax/6 * gs), gs = 448*6/amax) and the saturation rules are
 * the workload definitions that go with the pages' workloads.
 *
 * Arithmetic: IEEE-754 binary32, round-to-nearest-even, no FMA contraction
 * (built with -ffp-contract=off), subnormals kept.  Every step runs in the
 * order written below.  Readings of points the pages leave open:
 *  R1 RMSNorm normalises the T-rounded h (= residual_out), not the fp32 sum.
 *  R2 y stays fp32 (not rounded to T) before quantisation.
 *  R3 sum of squares: canonical pairwise tree (zero-pad to a power of two,
 *     add adjacent pairs level by level).
 *  R4 q = e4m3(y / s) with a correctly rounded fp32 division.
 *  R5 group scales are floored at 1e-12 like per-token scales.
 *  R6 NVFP4 global scale gs is an input; r = gs / decode(block scale) per
 *     block (0 when the block scale is 0); q = e2m1(y * r).
 *  R7 E2M1 nibble order: element 2j in the low nibble of byte j.
 *  R8 column-major group scales use stride n_tokens.
 *  R14 dynamic NVFP4 global scale: gs = 1 when amax over the batch is 0.
 *  R15 SiLU+Mul (vLLM docs, same page, section "SiLU+Mul + Quantization
 *      (fuse_act_quant)": silu_and_mul on the gated up-projection, then the
 *      quantisation, no full-precision activation tensor in between): each
 *      row of the input holds the gate g in its first d elements and the up
 *      projection u in the next d; silu(g) = g / (1 + e^-g) is its plain
 *      definition, evaluated in binary64 (the C library's exp) from the exact
 *      widening of g and rounded once to binary32; a = silu(g) * u is one
 *      binary32 product, kept in fp32 like y; then the same quantisation as
 *      the norm op.
 *  R16 (no exp routine of its own: the pages fix none, and the definition of
 *      silu above needs only the binary64 exponential.)
 *  R17 E8M0 scale option (blog, "Why this design", item 3: E8M0 scales,
 *      column-major scales and TMA alignment registered as combinable
 *      options): a dynamic (per-token or group) scale is rounded up to the
 *      next power of two, s = 2^ceil(log2 s), still stored as fp32 (its E8M0
 *      byte is the exponent field); q = e4m3(y / s) as before.
 *  R18 TMA-aligned option for column-major group scales: the stride between
 *      the scale columns of consecutive groups is n_tokens rounded up to a
 *      multiple of 4 (16 bytes); the padding entries are not written.
 *  R22 all-reduce + RMSNorm (vLLM docs, same page, section "AllReduce +
 *      RMSNorm (fuse_allreduce_rms)": the tensor-parallel all-reduce fused
 *      with the following residual add, RMSNorm and quantisation): the
 *      reduced activation is the rank-order binary32 sum of the ranks'
 *      partial tensors, rounded once to T; it is the x of the fused op.
 *  R21 UE8M0 byte option (the same item of the blog): the power-of-two scale
 *      of R17 is stored as one byte, its biased binary32 exponent (the UE8M0
 *      encoding: byte e stands for 2^(e - 127)), in the same layouts; with
 *      the TMA-aligned column layout the stride is n_tokens rounded up to 16
 *      (16 bytes).  Codes are those of R17.
 *  R19 the unfused sequence the fusion replaces (vLLM docs, same page,
 *      fuse_norm_quant: rms_norm / fused_add_rms_norm followed by quant_fp8):
 *      the first op writes y rounded to the activation type T (nearest even)
 *      and the updated residual; the second quantises that T tensor exactly
 *      as step 5 quantises y.
 *  R20 QK-norm + RoPE (vLLM docs, same page, section "QK Norm + RoPE
 *      (enable_qk_norm_rope_fusion)": split QKV, per-head RMSNorm of Q and K,
 *      rotary embedding, in one kernel): each q and k head of a token row is
 *      normalised like a row of the norm op (canonical sum over head_dim,
 *      inv = 1/sqrt(S/D + eps), y = (x * inv) * w with the q or k weight),
 *      kept in fp32, rotated with cos / sin taken from a caller-given fp32
 *      table [max_pos, D] (cos in the first D/2 columns, sin in the rest) at
 *      the token's position, each product and each sum rounded separately,
 *      and written back in place rounded once to T; v is untouched.  NeoX
 *      pairs element i with i + D/2, GPT-J pairs 2i with 2i+1 (both use
 *      angle index i).  A token whose position is outside [0, max_pos) is
 *      left unchanged.
 *  Parity unpinned: NaN / Inf inputs (IEEE propagation, not pinned by any test).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_BF16 = 0, OR_FP16 = 1 };
/* Option bits of the mode argument (R17, R18). */
enum { OR_OPT_E8M0 = 0x10, OR_OPT_TMA = 0x20, OR_OPT_UE8M0 = 0x40 };
enum {
    OR_FP8_STATIC = 0,
    OR_FP8_PER_TOKEN = 1,
    OR_FP8_G128_ROW = 2,
    OR_FP8_G128_COL = 3,
    OR_FP8_G64_ROW = 4,
    OR_FP8_G64_COL = 5,
    OR_NVFP4 = 6
};

/* ------------------------------------------------------------------------ */
/* Number formats, from their definitions.                                  */
/* ------------------------------------------------------------------------ */

static float bits_to_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t float_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the upper half of a binary32: widening is exact. */
float oracle_bf16_to_float(uint16_t b) { return bits_to_float((uint32_t)b << 16); }

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
float oracle_fp16_to_float(uint16_t b)
{
    int sign = b >> 15, e = (b >> 10) & 0x1f, m = b & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);                  /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + m), e - 25);      /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* binary32 -> bf16, round to nearest, ties to even on the 16 dropped bits. */
uint16_t oracle_float_to_bf16(float f)
{
    uint32_t u = float_to_bits(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    uint32_t upper = u >> 16, lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1; /* carry may reach inf */
    return (uint16_t)upper;
}

/* binary32 -> binary16, round to nearest even; overflow to +-inf. */
uint16_t oracle_float_to_fp16(float f)
{
    uint16_t sign = (uint16_t)(signbit(f) ? 0x8000 : 0);
    float a = fabsf(f);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7c00);   /* halfway 65504..65536 ties up to inf */
    if (a < ldexpf(1.0f, -14)) {                           /* subnormal range, step 2^-24 */
        float k = rintf(ldexpf(a, 24));                    /* exact scaling, RNE */
        return (uint16_t)(sign | (uint16_t)k);            /* k == 1024 is the smallest normal */
    }
    int ex;
    frexpf(a, &ex);                                        /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                                        /* a in [2^e, 2^(e+1)) */
    float k = rintf(ldexpf(a, 10 - e));                    /* significand * 1024 in [1024, 2048] */
    if (k == 2048.0f) { k = 1024.0f; e += 1; }
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)k - 1024));
}

/* OCP FP8 E4M3 (E4M3FN): bias 7, 3 fraction bits, no infinities, 0x7f/0xff
 * NaN, max 448, subnormals k * 2^-9.  Round to nearest even, saturate finite
 * and infinite magnitudes above 448 to 448, NaN -> 0x7f, sign always kept. */
uint8_t oracle_e4m3_encode(float v)
{
    if (isnan(v)) return 0x7f;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    float a = fabsf(v);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7e);
    if (a < ldexpf(1.0f, -6)) {                            /* subnormal range, step 2^-9 */
        float k = rintf(ldexpf(a, 9));                     /* 0..8; 8 is the smallest normal */
        return (uint8_t)(sign | (uint8_t)k);
    }
    int ex;
    frexpf(a, &ex);
    int e = ex - 1;
    float k = rintf(ldexpf(a, 3 - e));                     /* in [8, 16] */
    if (k == 16.0f) { k = 8.0f; e += 1; }
    int code = ((e + 7) << 3) | ((int)k - 8);
    if (code > 0x7e) code = 0x7e;
    return (uint8_t)(sign | code);
}

float oracle_e4m3_decode(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 0xf, m = c & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexpf((float)m, -9);
    else v = ldexpf((float)(8 + m), e - 10);               /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* FP4 E2M1: bias 1, 1 fraction bit: {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  Round to
 * nearest even, saturate to 6, sign always kept (-0 -> 0x8). */
uint8_t oracle_e2m1_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    float a = fabsf(v);
    if (isnan(v)) return 0x7;      /* not reached by the tests (NaN is out of scope) */
    if (a >= 6.0f) return (uint8_t)(sign | 0x7);
    if (a < 1.0f) {                                        /* subnormal range, step 0.5 */
        float k = rintf(a * 2.0f);                         /* 0, 1, 2; 2 is 1.0 */
        return (uint8_t)(sign | (uint8_t)k);
    }
    int ex;
    frexpf(a, &ex);
    int e = ex - 1;                                        /* 0, 1 or 2 */
    float k = rintf(ldexpf(a, 1 - e));                     /* in [2, 4] */
    if (k == 4.0f) { k = 2.0f; e += 1; }
    int code = ((e + 1) << 1) | ((int)k - 2);
    if (code > 7) code = 7;
    return (uint8_t)(sign | code);
}

float oracle_e2m1_decode(uint8_t c)
{
    int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    float v = (e == 0) ? 0.5f * (float)m : ldexpf((float)(2 + m), e - 2);
    return sign ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* silu (reading R15).                                                      */
/* ------------------------------------------------------------------------ */

/* silu(g) = g / (1 + e^-g), in binary64 from the exact widening of g, rounded
 * once to binary32.  The binary64 evaluation carries about 2^-52 relative
 * error, far below the binary32 rounding.  Non-finite g is outside the
 * readings (R13). */
float oracle_silu(float g)
{
    const double gd = (double)g;
    return (float)(gd / (1.0 + exp(-gd)));
}

/* ------------------------------------------------------------------------ */
/* Canonical pairwise sum (reading R3).                                     */
/* ------------------------------------------------------------------------ */

/* Zero-pad v[0..n) to P = next power of two >= n, then replace the sequence by
 * the sums of adjacent pairs (v[2k] + v[2k+1]) until one value is left.
 * buf must hold P floats. */
float oracle_tree_sum_buf(const float *v, int64_t n, float *buf)
{
    if (n <= 0) return 0.0f;
    int64_t P = 1;
    while (P < n) P <<= 1;
    for (int64_t i = 0; i < P; ++i) buf[i] = (i < n) ? v[i] : 0.0f;
    for (int64_t len = P; len > 1; len >>= 1)
        for (int64_t k = 0; k < len / 2; ++k) buf[k] = buf[2 * k] + buf[2 * k + 1];
    return buf[0];
}

float oracle_tree_sum(const float *v, int64_t n)
{
    int64_t P = 1;
    while (P < n) P <<= 1;
    float *buf = (float *)malloc((size_t)P * sizeof(float));
    float s = oracle_tree_sum_buf(v, n, buf);
    free(buf);
    return s;
}

/* ------------------------------------------------------------------------ */
/* The op, one row at a time.                                               */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *x, *residual, *weight;
    float eps;
    int mode;                /* base mode, without option bits */
    float scale_in;          /* FP8 static: s;  NVFP4: global scale gs */
    uint8_t *out_q;
    void *out_scales;
    uint16_t *residual_out;
    float *y_out;            /* optional fp32 copy of y [n, H] for diagnostics */
    int64_t n, H;
    int dtype;
    int silu_mul;            /* 1: the SiLU+Mul op, x = [n, 2H] gate | up (R15);
                                2: quantisation of x alone (R19) */
    uint16_t *y_t_out;       /* R19: y rounded to T instead of step 5 */
    int e8m0;                /* R17: 1 = power-of-two fp32 scales; R21: 2 = their UE8M0 bytes */
    int64_t col_stride;      /* column-major scale stride: n, or n rounded up to 4 (R18) */
    const float *y_in;       /* silu_mul == 3: step 5 alone on these fp32 rows [n, H] */
} OracleArgs;

/* The smallest power of two >= x, for a positive normal x: x = f 2^k with
 * f in [0.5, 1); 2^(k-1) when f = 0.5, else 2^k (exact). */
static float pow2_ceil(float x)
{
    int k;
    const float f = frexpf(x, &k);
    return f == 0.5f ? x : ldexpf(1.0f, k);
}

/* Mode argument -> base mode and options; -1 for an invalid combination. */
static int split_mode(int mode, int64_t n, int *base, int *e8m0, int64_t *col_stride)
{
    *base = mode & 0xf;
    const int opts = mode & ~0xf;
    if (*base < 0 || *base > 6 || (opts & ~(OR_OPT_E8M0 | OR_OPT_TMA | OR_OPT_UE8M0))) return -1;
    const int dynamic = *base >= OR_FP8_PER_TOKEN && *base <= OR_FP8_G64_COL;
    const int col = *base == OR_FP8_G128_COL || *base == OR_FP8_G64_COL;
    if ((opts & (OR_OPT_E8M0 | OR_OPT_UE8M0)) && !dynamic) return -1;
    if ((opts & OR_OPT_TMA) && !col) return -1;
    *e8m0 = (opts & OR_OPT_UE8M0) ? 2 : (opts & OR_OPT_E8M0) != 0;
    /* R18 / R21: 16 bytes between scale columns: 4 fp32 scales or 16 UE8M0 bytes */
    const int64_t per16 = (opts & OR_OPT_UE8M0) ? 16 : 4;
    *col_stride = (opts & OR_OPT_TMA) ? (n + per16 - 1) / per16 * per16 : n;
    return 0;
}

typedef struct {
    float *h, *sq, *y, *buf;
} RowScratch;

static float widen(int dtype, uint16_t b)
{
    return dtype == OR_BF16 ? oracle_bf16_to_float(b) : oracle_fp16_to_float(b);
}

static uint16_t narrow(int dtype, float f)
{
    return dtype == OR_BF16 ? oracle_float_to_bf16(f) : oracle_float_to_fp16(f);
}

static int group_size(int mode)
{
    switch (mode) {
    case OR_FP8_G128_ROW: case OR_FP8_G128_COL: return 128;
    case OR_FP8_G64_ROW: case OR_FP8_G64_COL: return 64;
    default: return 0;
    }
}

/* A dynamic scale into element i of the scale tensor: fp32, or with the
 * UE8M0 byte option (R21) the biased exponent of the power-of-two scale,
 * bits 30..23 of its binary32 pattern (byte e stands for 2^(e - 127)). */
static void store_scale(const OracleArgs *a, int64_t i, float sc)
{
    if (a->e8m0 == 2) {
        uint32_t u;
        memcpy(&u, &sc, 4);
        ((uint8_t *)a->out_scales)[i] = (uint8_t)((u >> 23) & 0xffu);
    } else {
        ((float *)a->out_scales)[i] = sc;
    }
}

/* Step 5 of the op: quantisation of the fp32 row y (R4-R8). */
static void quantize_row(const OracleArgs *a, int64_t t, const float *y)
{
    const int64_t H = a->H;
    uint8_t *q = a->out_q;
    if (a->mode == OR_FP8_STATIC) {
        float sc = a->scale_in;
        for (int64_t i = 0; i < H; ++i) q[t * H + i] = oracle_e4m3_encode(y[i] / sc);
    } else if (a->mode == OR_FP8_PER_TOKEN) {
        float amax = 0.0f;
        for (int64_t i = 0; i < H; ++i) amax = fmaxf(amax, fabsf(y[i]));
        float sc = fmaxf(amax / 448.0f, 1e-12f);
        if (a->e8m0) sc = pow2_ceil(sc);
        store_scale(a, t, sc);
        for (int64_t i = 0; i < H; ++i) q[t * H + i] = oracle_e4m3_encode(y[i] / sc);
    } else if (a->mode == OR_NVFP4) {
        float gs = a->scale_in;
        uint8_t *bs = (uint8_t *)a->out_scales;
        for (int64_t b = 0; b < H / 16; ++b) {
            const float *yb = y + 16 * b;
            float amax = 0.0f;
            for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(yb[k]));
            uint8_t sb = oracle_e4m3_encode((amax / 6.0f) * gs);
            bs[t * (H / 16) + b] = sb;
            float d = oracle_e4m3_decode(sb);
            float r = (d == 0.0f) ? 0.0f : gs / d;
            for (int k = 0; k < 16; k += 2) {
                uint8_t lo = oracle_e2m1_encode(yb[k] * r);
                uint8_t hi = oracle_e2m1_encode(yb[k + 1] * r);
                q[t * (H / 2) + 8 * b + k / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    } else {
        int G = group_size(a->mode);
        int col = (a->mode == OR_FP8_G128_COL || a->mode == OR_FP8_G64_COL);
        for (int64_t g = 0; g < H / G; ++g) {
            const float *yg = y + G * g;
            float amax = 0.0f;
            for (int k = 0; k < G; ++k) amax = fmaxf(amax, fabsf(yg[k]));
            float sc = fmaxf(amax / 448.0f, 1e-12f);
            if (a->e8m0) sc = pow2_ceil(sc);
            store_scale(a, col ? g * a->col_stride + t : t * (H / G) + g, sc);
            for (int k = 0; k < G; ++k) q[t * H + G * g + k] = oracle_e4m3_encode(yg[k] / sc);
        }
    }
}

static void oracle_row(const OracleArgs *a, int64_t t, RowScratch *s)
{
    const int64_t H = a->H;
    const uint16_t *xr = a->x + t * H;

    /* Step 1: residual add, h rounded to the activation type and written back
     * as the updated residual (R1); without a residual, h = x. */
    for (int64_t i = 0; i < H; ++i) {
        if (a->residual) {
            float sum = widen(a->dtype, xr[i]) + widen(a->dtype, a->residual[t * H + i]);
            uint16_t hb = narrow(a->dtype, sum);
            a->residual_out[t * H + i] = hb;
            s->h[i] = widen(a->dtype, hb);
        } else {
            s->h[i] = widen(a->dtype, xr[i]);
        }
    }

    /* Step 2: sum of squares by the canonical tree (R3). */
    for (int64_t i = 0; i < H; ++i) s->sq[i] = s->h[i] * s->h[i];
    float S = oracle_tree_sum_buf(s->sq, H, s->buf);

    /* Step 3: mean square and reciprocal RMS, each correctly rounded. */
    float ms = S / (float)H;
    float inv = 1.0f / sqrtf(ms + a->eps);

    /* Step 4: y = (h * inv) * w, kept in fp32 (R2). */
    for (int64_t i = 0; i < H; ++i)
        s->y[i] = (s->h[i] * inv) * widen(a->dtype, a->weight[i]);
    if (a->y_out) memcpy(a->y_out + t * H, s->y, (size_t)H * sizeof(float));
    if (a->y_t_out) {   /* R19: the unfused first op ends here */
        for (int64_t i = 0; i < H; ++i) a->y_t_out[t * H + i] = narrow(a->dtype, s->y[i]);
        return;
    }

    /* Step 5: quantisation. */
    quantize_row(a, t, s->y);
}

/* R19, second op: step 5 on a T row. */
static void oracle_quant_row(const OracleArgs *a, int64_t t, RowScratch *s)
{
    for (int64_t i = 0; i < a->H; ++i) s->y[i] = widen(a->dtype, a->x[t * a->H + i]);
    quantize_row(a, t, s->y);
}

/* SiLU+Mul, one row (R15): a = silu(g) * u in fp32, then step 5 of the norm
 * op on a. */
static void oracle_act_row(const OracleArgs *a, int64_t t, RowScratch *s)
{
    const int64_t d = a->H;
    const uint16_t *g = a->x + t * 2 * d, *u = g + d;
    for (int64_t i = 0; i < d; ++i)
        s->y[i] = oracle_silu(widen(a->dtype, g[i])) * widen(a->dtype, u[i]);
    if (a->y_out) memcpy(a->y_out + t * d, s->y, (size_t)d * sizeof(float));
    quantize_row(a, t, s->y);
}

typedef struct {
    const OracleArgs *a;
    int64_t r0, r1;
    int ok;
} Span;

static void *run_span(void *p)
{
    Span *sp = (Span *)p;
    int64_t H = sp->a->H, P = 1;
    while (P < H) P <<= 1;
    RowScratch s;
    s.h = (float *)malloc((size_t)H * sizeof(float));
    s.sq = (float *)malloc((size_t)H * sizeof(float));
    s.y = (float *)malloc((size_t)H * sizeof(float));
    s.buf = (float *)malloc((size_t)P * sizeof(float));
    sp->ok = s.h && s.sq && s.y && s.buf;
    if (sp->ok)
        for (int64_t t = sp->r0; t < sp->r1; ++t) {
            if (sp->a->silu_mul == 3) quantize_row(sp->a, t, sp->a->y_in + t * H);
            else if (sp->a->silu_mul == 2) oracle_quant_row(sp->a, t, &s);
            else if (sp->a->silu_mul) oracle_act_row(sp->a, t, &s);
            else oracle_row(sp->a, t, &s);
        }
    free(s.h); free(s.sq); free(s.y); free(s.buf);
    return NULL;
}

static int run_rows(const OracleArgs *ap, int nthreads);

/* Whole tensor.  Returns 0 on success, -1 on a bad argument, -2 on an
 * allocation or thread failure. */
int oracle_fused_add_rmsnorm_quant(const uint16_t *x, const uint16_t *residual,
                                   const uint16_t *weight, float eps, int mode, float scale_in,
                                   uint8_t *out_q, void *out_scales, uint16_t *residual_out,
                                   float *y_out, int64_t n, int64_t H, int dtype, int nthreads)
{
    int e8m0;
    int64_t col_stride;
    if (n < 0 || split_mode(mode, n, &mode, &e8m0, &col_stride)) return -1;
    if (H <= 0 || (dtype != OR_BF16 && dtype != OR_FP16)) return -1;
    if (!x || !weight || !out_q || (residual && !residual_out)) return -1;
    if (mode != OR_FP8_STATIC && !out_scales) return -1;
    if (mode == OR_NVFP4 && H % 16) return -1;
    if (group_size(mode) && H % group_size(mode)) return -1;
    OracleArgs a = {x, residual, weight, eps, mode, scale_in, out_q, out_scales,
                    residual_out, y_out, n, H, dtype, 0, NULL, e8m0, col_stride};
    return run_rows(&a, nthreads);
}

/* Rows are independent, so splitting them over threads gives bit-identical
 * results for any thread count. */
static int run_rows(const OracleArgs *ap, int nthreads)
{
    const OracleArgs a = *ap;
    const int64_t n = a.n;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    Span *spans = (Span *)calloc((size_t)nthreads, sizeof(Span));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!spans || !th) { free(spans); free(th); return -2; }
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        spans[i].a = &a;
        spans[i].r0 = n * i / nthreads;
        spans[i].r1 = n * (i + 1) / nthreads;
    }
    if (nthreads == 1) {
        run_span(&spans[0]);
    } else {
        int started = 0;
        for (; started < nthreads; ++started)
            if (pthread_create(&th[started], NULL, run_span, &spans[started])) break;
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        if (started < nthreads) rc = -2;
    }
    for (int i = 0; i < nthreads && !rc; ++i)
        if (!spans[i].ok) rc = -2;
    free(spans);
    free(th);
    return rc;
}

/* SiLU+Mul + quantisation (R15): gate_up [n, 2d] (gate | up per row), the
 * quantisation of `mode` on a = silu(gate) * up; y_out (optional) receives a.
 * Returns 0, or -1 / -2 like oracle_fused_add_rmsnorm_quant. */
int oracle_silu_mul_quant(const uint16_t *gate_up, int mode, float scale_in, uint8_t *out_q,
                          void *out_scales, float *y_out, int64_t n, int64_t d, int dtype, int nthreads)
{
    int e8m0;
    int64_t col_stride;
    if (n < 0 || split_mode(mode, n, &mode, &e8m0, &col_stride)) return -1;
    if (d <= 0 || (dtype != OR_BF16 && dtype != OR_FP16)) return -1;
    if (!gate_up || !out_q || (mode != OR_FP8_STATIC && !out_scales)) return -1;
    if (mode == OR_NVFP4 && d % 16) return -1;
    if (group_size(mode) && d % group_size(mode)) return -1;
    OracleArgs a = {gate_up, NULL, NULL, 0.0f, mode, scale_in, out_q, out_scales,
                    NULL, y_out, n, d, dtype, 1, NULL, e8m0, col_stride};
    return run_rows(&a, nthreads);
}

/* R22: all-reduce + residual add + RMSNorm + quantisation.  partials holds
 * nranks [n, H] tensors one after the other; x = T(sum of their widened
 * values in rank order, binary32), then the fused op on x.  Returns 0, or -1
 * / -2 like oracle_fused_add_rmsnorm_quant. */
int oracle_allreduce_add_rmsnorm_quant(const uint16_t *partials, int nranks, const uint16_t *residual,
                                       const uint16_t *weight, float eps, int mode, float scale_in,
                                       uint8_t *out_q, void *out_scales, uint16_t *residual_out, float *y_out,
                                       int64_t n, int64_t H, int dtype, int nthreads)
{
    if (!partials || nranks < 1 || n < 0 || H <= 0 || (dtype != OR_BF16 && dtype != OR_FP16)) return -1;
    uint16_t *x = (uint16_t *)malloc((size_t)(n * H > 0 ? n * H : 1) * sizeof(uint16_t));
    if (!x) return -2;
    for (int64_t i = 0; i < n * H; ++i) {
        float acc = widen(dtype, partials[i]);
        for (int r = 1; r < nranks; ++r) acc = acc + widen(dtype, partials[(int64_t)r * n * H + i]);
        x[i] = narrow(dtype, acc);
    }
    const int rc = oracle_fused_add_rmsnorm_quant(x, residual, weight, eps, mode, scale_in, out_q, out_scales,
                                                  residual_out, y_out, n, H, dtype, nthreads);
    free(x);
    return rc;
}

/* Step 5 alone (R4-R8, R17, R18) on given fp32 rows y [n, d]: the
 * quantisation any producer of fp32 activations feeds.  Returns 0, or -1 /
 * -2 like oracle_fused_add_rmsnorm_quant. */
int oracle_quant_f32(const float *y, int mode, float scale_in, uint8_t *out_q, void *out_scales, int64_t n,
                     int64_t d, int nthreads)
{
    int e8m0;
    int64_t col_stride;
    if (n < 0 || split_mode(mode, n, &mode, &e8m0, &col_stride)) return -1;
    if (d <= 0 || !y || !out_q || (mode != OR_FP8_STATIC && !out_scales)) return -1;
    if (mode == OR_NVFP4 && d % 16) return -1;
    if (group_size(mode) && d % group_size(mode)) return -1;
    OracleArgs a = {NULL, NULL, NULL, 0.0f, mode, scale_in, out_q, out_scales,
                    NULL, NULL, n, d, OR_BF16, 3, NULL, e8m0, col_stride, y};
    return run_rows(&a, nthreads);
}

/* R20: QK-norm + RoPE, in place on qkv [n, (nq + 2 nkv) D] (q heads, then k
 * heads, then v heads of each token).  Returns 0, or -1 on a bad argument. */
static void norm_rope_head(uint16_t *head, const uint16_t *w, float eps, const float *cs, int D, int neox,
                           int dtype, float *x, float *sq, float *buf, float *y)
{
    for (int i = 0; i < D; ++i) { x[i] = widen(dtype, head[i]); sq[i] = x[i] * x[i]; }
    const float S = oracle_tree_sum_buf(sq, D, buf);
    const float inv = 1.0f / sqrtf(S / (float)D + eps);
    for (int i = 0; i < D; ++i) y[i] = (x[i] * inv) * widen(dtype, w[i]);
    const int h = D / 2;
    for (int i = 0; i < h; ++i) {
        const float c = cs[i], s = cs[h + i];
        const int a = neox ? i : 2 * i, b = neox ? i + h : 2 * i + 1;
        const float ya = y[a], yb = y[b];
        const float oa = ya * c - yb * s;
        const float ob = yb * c + ya * s;
        head[a] = narrow(dtype, oa);
        head[b] = narrow(dtype, ob);
    }
}

int oracle_qk_norm_rope(uint16_t *qkv, const int64_t *positions, const float *cos_sin, int64_t max_pos,
                        const uint16_t *q_w, const uint16_t *k_w, float eps, int64_t n, int nq, int nkv, int D,
                        int neox, int dtype)
{
    if (n < 0 || nq < 0 || nkv < 0 || D <= 0 || D % 2 || (dtype != OR_BF16 && dtype != OR_FP16)) return -1;
    if (!qkv || !positions || !cos_sin || !q_w || !k_w || max_pos <= 0) return -1;
    float *tmp = (float *)malloc((size_t)D * 4 * sizeof(float) + 8 * sizeof(float) * (size_t)D);
    if (!tmp) return -2;
    float *x = tmp, *sq = tmp + D, *y = tmp + 2 * D, *buf = tmp + 3 * D;
    const int64_t width = (int64_t)(nq + 2 * nkv) * D;
    for (int64_t t = 0; t < n; ++t) {
        const int64_t pos = positions[t];
        if (pos < 0 || pos >= max_pos) continue;
        const float *cs = cos_sin + pos * D;
        for (int hd = 0; hd < nq + nkv; ++hd)
            norm_rope_head(qkv + t * width + (int64_t)hd * D, hd < nq ? q_w : k_w, eps, cs, D, neox, dtype,
                           x, sq, buf, y);
    }
    free(tmp);
    return 0;
}

/* R19: the two ops of the unfused sequence.  oracle_add_rmsnorm writes y
 * rounded to T into y_t [n, H] (and residual_out); oracle_quant quantises a T
 * tensor [n, H] by `mode`.  Returns like oracle_fused_add_rmsnorm_quant. */
int oracle_add_rmsnorm(const uint16_t *x, const uint16_t *residual, const uint16_t *weight, float eps,
                       uint16_t *y_t, uint16_t *residual_out, int64_t n, int64_t H, int dtype, int nthreads)
{
    if (n < 0 || H <= 0 || (dtype != OR_BF16 && dtype != OR_FP16)) return -1;
    if (!x || !weight || !y_t || (residual && !residual_out)) return -1;
    OracleArgs a = {x, residual, weight, eps, OR_FP8_STATIC, 0.0f, NULL, NULL,
                    residual_out, NULL, n, H, dtype, 0, y_t, 0, n};
    return run_rows(&a, nthreads);
}

int oracle_quant(const uint16_t *y_t, int mode, float scale_in, uint8_t *out_q, void *out_scales,
                 int64_t n, int64_t H, int dtype, int nthreads)
{
    int e8m0;
    int64_t col_stride;
    if (n < 0 || split_mode(mode, n, &mode, &e8m0, &col_stride)) return -1;
    if (H <= 0 || (dtype != OR_BF16 && dtype != OR_FP16)) return -1;
    if (!y_t || !out_q || (mode != OR_FP8_STATIC && !out_scales)) return -1;
    if (mode == OR_NVFP4 && H % 16) return -1;
    if (group_size(mode) && H % group_size(mode)) return -1;
    OracleArgs a = {y_t, NULL, NULL, 0.0f, mode, scale_in, out_q, out_scales,
                    NULL, NULL, n, H, dtype, 2, NULL, e8m0, col_stride};
    return run_rows(&a, nthreads);
}

void oracle_silu_array(const float *v, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_silu(v[i]);
}

/* NVFP4 with the global scale taken from the data: gs = 448 * 6 / amax over
 * every y of the batch (the NVFP4 workload's definition of the global scale),
 * reading R14: gs = 1 when that amax is 0 (an all-zero batch).  First pass: the
 * op up to y for every row (residual written back) and the batch amax; second
 * pass: the NVFP4 quantisation of y with that gs.  *out_gs receives gs.
 * Returns 0, or -1 / -2 like oracle_fused_add_rmsnorm_quant. */
int oracle_fused_add_rmsnorm_nvfp4_dynamic(const uint16_t *x, const uint16_t *residual,
                                           const uint16_t *weight, float eps, uint8_t *out_q,
                                           uint8_t *out_block_scales, float *out_gs,
                                           uint16_t *residual_out, int64_t n, int64_t H, int dtype,
                                           int nthreads)
{
    if (n < 0 || H <= 0 || H % 16 || !out_gs) return -1;
    float *y = (float *)malloc((size_t)(n > 0 ? n : 1) * (size_t)H * sizeof(float));
    if (!y) return -2;
    /* pass 1: per-token FP8 run, only for its y (codes and scales discarded) */
    uint8_t *tmp_q = (uint8_t *)malloc((size_t)(n > 0 ? n : 1) * (size_t)H);
    float *tmp_s = (float *)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    int rc = (tmp_q && tmp_s) ? 0 : -2;
    if (!rc)
        rc = oracle_fused_add_rmsnorm_quant(x, residual, weight, eps, OR_FP8_PER_TOKEN, 0.0f, tmp_q,
                                            tmp_s, residual_out, y, n, H, dtype, nthreads);
    float amax = 0.0f;
    for (int64_t i = 0; !rc && i < n * H; ++i) amax = fmaxf(amax, fabsf(y[i]));
    float gs = (amax > 0.0f) ? 2688.0f / amax : 1.0f;
    /* pass 2: NVFP4 with gs, on the same inputs (y is recomputed identically) */
    if (!rc)
        rc = oracle_fused_add_rmsnorm_quant(x, residual, weight, eps, OR_NVFP4, gs, out_q,
                                            out_block_scales, residual_out, NULL, n, H, dtype,
                                            nthreads);
    if (!rc) *out_gs = gs;
    free(y);
    free(tmp_q);
    free(tmp_s);
    return rc;
}

/* Array forms of the codecs, for exhaustive checks. */
void oracle_e4m3_encode_array(const float *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e2m1_encode_array(const float *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(v[i]);
}

void oracle_float_to_bf16_array(const float *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_float_to_bf16(v[i]);
}

void oracle_float_to_fp16_array(const float *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_float_to_fp16(v[i]);
}

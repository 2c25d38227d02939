/*
 * librmsq — fused residual-add + RMSNorm + activation quantisation on GB300 (sm_103a).
 *
 * The operation is the one vLLM's RMSNorm + quantisation fusion puts in place
 * of a separate (fused-add) RMSNorm kernel and a quantisation kernel:
 *   vLLM docs, "Fusion torch.compile passes", section
 *   "RMSNorm + Quantization (fuse_norm_quant)": rms_norm(x) -> quant_fp8(y) and
 *   fused_add_rms_norm(x, residual) -> quant_fp8(y), the residual updated in
 *   place; schemes FP8 static per-tensor, FP8 dynamic per-token and FP8
 *   dynamic per-token-group (128/64);
 *   blog "[vLLM] Compilation Fusion Passes", sections "Pattern matching
 *   structure" (result, input, weight, scale, epsilon), "Fused Add + RMSNorm +
 *   Group Quantization" (the fused-op table keyed by quant scheme and fused
 *   add), "Type validation" (input and weight share one dtype) and "Why this
 *   design" (column-major scales);
 *   vLLM PR #51925 summary (prhub), "Motivation" and "Key source snippets":
 *   residual update + RMSNorm followed by NVFP4 block scales and FP4 values,
 *   with an fp32 activation (global) scale given as an input.
 *
 * Per row t of an [n_tokens, hidden] activation (T = bf16 or fp16):
 *   h    = T(fp32(x) + fp32(residual))       (h = x when residual is NULL)
 *   residual_out = h
 *   S    = pairwise-tree sum of fp32(h)^2     (zero-pad to a power of two,
 *                                              add adjacent pairs level by level)
 *   inv  = 1 / sqrt(S / hidden + eps)         (IEEE division and square root)
 *   y    = (fp32(h) * inv) * fp32(weight)     (fp32, not rounded to T)
 *   then one of the quantisation modes below.  All fp32 arithmetic rounds to
 *   nearest even; results are bit-identical to that definition.
 *
 * Besides that op (rmsq_fused_add_rmsnorm_quant and its variants) the library
 * has: NVFP4 with the global scale taken from the data
 * (rmsq_fused_add_rmsnorm_nvfp4_dynamic); scale options E8M0 and TMA-aligned
 * column-major (RMSQ_QUANT_*); SiLU+Mul + quantisation (rmsq_silu_mul_quant,
 * the same docs page's "SiLU+Mul + Quantization (fuse_act_quant)"); and the
 * unfused two-op sequence the fusion replaces (rmsq_fused_add_rmsnorm,
 * rmsq_quant); and QK-norm + RoPE on the attention input
 * (rmsq_qk_norm_rope, the docs page's "QK Norm + RoPE
 * (enable_qk_norm_rope_fusion)").
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" must be addressable by the current CUDA device
 *     (cudaMalloc / torch CUDA tensors, or managed memory).  The caller owns
 *     every buffer; the library allocates no device memory and keeps no
 *     per-call state.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous with respect to the host and do not synchronise.
 *   - Argument errors are reported synchronously, before any launch, and leave
 *     every output untouched.  A failed launch returns RMSQ_ERR_CUDA; the CUDA
 *     error code is then available from rmsq_last_cuda_error().
 *   - Device code is built for sm_103a only; any other device gives
 *     RMSQ_ERR_UNSUPPORTED_DEVICE and there is no CPU fallback.
 */
#ifndef RMSQ_H
#define RMSQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RMSQ_VERSION 10000        /* 1.0.0 */
#define RMSQ_MAX_HIDDEN 16384

typedef enum {
    RMSQ_OK = 0,
    RMSQ_ERR_INVALID_ARG = 1,        /* NULL where a pointer is required, bad enum, bad eps */
    RMSQ_ERR_ALIGNMENT = 2,          /* a pointer misses the alignment stated below */
    RMSQ_ERR_ALIAS = 3,              /* outputs overlap inputs other than as allowed */
    RMSQ_ERR_UNSUPPORTED_SHAPE = 4,  /* hidden not a multiple of 8 / the group / 16, or too large */
    RMSQ_ERR_UNSUPPORTED_DEVICE = 5, /* current device is not compute capability 10.3 */
    RMSQ_ERR_NO_DEVICE = 6,          /* no CUDA device / driver */
    RMSQ_ERR_CUDA = 7                /* a CUDA runtime call or launch failed */
} rmsq_status;

typedef enum { RMSQ_BF16 = 0, RMSQ_FP16 = 1 } rmsq_dtype;

/*
 * Quantisation modes (blog "[vLLM] Compilation Fusion Passes", section
 * "Fused Add + RMSNorm + Group Quantization": static per-tensor, dynamic
 * per-token and dynamic 128-group symmetric FP8; vLLM docs "Fusion
 * torch.compile passes", fuse_norm_quant: group 128 or 64; PR #51925: NVFP4).
 * E4M3 is OCP FP8 E4M3FN: round to nearest even, magnitudes above 448
 * (including infinities) saturate to 448, sign kept (-0 -> 0x80).
 *
 *  RMSQ_FP8_STATIC        s = scale_in[0];                q = e4m3(y / s)
 *  RMSQ_FP8_PER_TOKEN     s_t = max(amax_t(|y|) / 448, 1e-12), fp32 [n_tokens]
 *  RMSQ_FP8_GROUP{128,64}_ROW  s_{t,g} over G contiguous elements, fp32 [n_tokens, hidden/G]
 *  RMSQ_FP8_GROUP{128,64}_COL  same values stored [hidden/G, n_tokens] (column-major)
 *                         q = e4m3(y / s), one byte per element, [n_tokens, hidden]
 *  RMSQ_NVFP4             per 16-element block b: sb = e4m3((amax_b / 6) * gs),
 *                         gs = scale_in[0]; d = decode(sb); r = d ? gs / d : 0;
 *                         q = e2m1(y * r) (values {0,.5,1,1.5,2,3,4,6}, round to
 *                         nearest even, saturate at 6, sign kept); element 2j in
 *                         the low nibble of byte j: q is u8 [n_tokens, hidden/2],
 *                         block scales u8 (E4M3) [n_tokens, hidden/16], row-major.
 * The divisions y / s are correctly rounded fp32 divisions.
 */
typedef enum {
    RMSQ_FP8_STATIC = 0,
    RMSQ_FP8_PER_TOKEN = 1,
    RMSQ_FP8_GROUP128_ROW = 2,
    RMSQ_FP8_GROUP128_COL = 3,
    RMSQ_FP8_GROUP64_ROW = 4,
    RMSQ_FP8_GROUP64_COL = 5,
    RMSQ_NVFP4 = 6
} rmsq_quant_mode;

/*
 * Scale options, OR-ed into a quant_mode argument (blog "[vLLM] Compilation
 * Fusion Passes", section "Why this design", item 3: E8M0 scales,
 * column-major scales and TMA alignment registered as combinable options).
 *  RMSQ_QUANT_E8M0         the dynamic scale (per-token and group modes only)
 *                          is rounded up to a power of two,
 *                          s = 2^ceil(log2 max(amax / 448, 1e-12)); it is
 *                          still stored as fp32 (its E8M0 byte is the
 *                          exponent field, bits 30..23), q = e4m3(y / s).
 *  RMSQ_QUANT_UE8M0        the same power-of-two scale, stored as one byte
 *                          (per-token and group modes only): the UE8M0
 *                          encoding, byte e standing for 2^(e - 127) (the
 *                          biased exponent of the fp32 scale).  out_scales is
 *                          then u8 with the layouts below (1-byte aligned);
 *                          implies RMSQ_QUANT_E8M0, codes are the same.
 *  RMSQ_QUANT_TMA_ALIGNED  column-major group scales (_COL modes only) use a
 *                          stride of n_tokens rounded up to 16 bytes of scales
 *                          between groups: [hidden/G, round4(n)] fp32 scales,
 *                          or [hidden/G, round16(n)] UE8M0 bytes; the padding
 *                          entries are not written.
 * Any other bit, or an option with a mode it does not apply to, is
 * RMSQ_ERR_INVALID_ARG.
 */
#define RMSQ_QUANT_MODE_MASK 0x0f
#define RMSQ_QUANT_E8M0 0x10
#define RMSQ_QUANT_TMA_ALIGNED 0x20
#define RMSQ_QUANT_UE8M0 0x40

/*
 * rmsq_fused_add_rmsnorm_quant — one launch of the fused op over n_tokens rows.
 *
 *  x            device, T[n_tokens, hidden], row-major, 16-byte aligned.
 *  residual     device, T[n_tokens, hidden], 16-byte aligned, or NULL (plain
 *               RMSNorm + quant: h = x, nothing is written to residual_out).
 *  weight       device, T[hidden], 16-byte aligned (same dtype as x).
 *  eps          finite, >= 0 (1e-5 and 1e-6 are the values the pages use).
 *  quant_mode   an rmsq_quant_mode, optionally OR-ed with RMSQ_QUANT_* options.
 *  scale_in     device, one fp32: the static scale s (FP8_STATIC) or the global
 *               scale gs (NVFP4); ignored (may be NULL) for the dynamic FP8
 *               modes.  Its value must be finite and > 0; it is not checked.
 *  out_q        device, u8[n_tokens, hidden] (FP8) or u8[n_tokens, hidden/2]
 *               (NVFP4), 16-byte aligned.
 *  out_scales   device; fp32 per-token / per-group scales (4-byte aligned),
 *               their UE8M0 bytes (RMSQ_QUANT_UE8M0), or u8 NVFP4 block
 *               scales; ignored (may be NULL) for FP8_STATIC.
 *               rmsq_query_sizes gives the byte sizes.
 *  residual_out device, T[n_tokens, hidden], 16-byte aligned; NULL exactly when
 *               residual is NULL.  It may be the same pointer as residual (the
 *               in-place update of fused_add_rms_norm) or as x.
 *  n_tokens     >= 0 and < 2^31; 0 returns RMSQ_OK without a launch.
 *  hidden       > 0, a multiple of 8 (16 for NVFP4, G for the group modes),
 *               <= RMSQ_MAX_HIDDEN.
 *  dtype        an rmsq_dtype: the type of x, residual, weight, residual_out.
 *  stream       cudaStream_t to launch on.
 * Aliasing: besides residual_out == residual or residual_out == x, no output
 * may overlap any input or another output, and x / residual / residual_out
 * must be identical or disjoint.
 * Returns an rmsq_status.
 */
int rmsq_fused_add_rmsnorm_quant(const void *x, const void *residual, const void *weight,
                                 float eps, int quant_mode, const float *scale_in,
                                 void *out_q, void *out_scales, void *residual_out,
                                 int64_t n_tokens, int64_t hidden, int dtype, void *stream);

/*
 * Kernel variants.  Both compute bit-identical results; AUTO picks by batch
 * size.  DIRECT: one CTA per row, loads straight into registers (lowest
 * latency for a few rows).  PIPELINED: persistent CTAs with several rows per
 * CTA in flight as bulk asynchronous copies into shared memory (highest
 * bandwidth for large batches).
 */
typedef enum { RMSQ_VARIANT_AUTO = 0, RMSQ_VARIANT_DIRECT = 1, RMSQ_VARIANT_PIPELINED = 2 } rmsq_variant;

/*
 * rmsq_fused_add_rmsnorm_quant_ex — rmsq_fused_add_rmsnorm_quant with an
 * explicit rmsq_variant (RMSQ_ERR_INVALID_ARG for any other value).  Same
 * arguments, rules and results otherwise.
 */
int rmsq_fused_add_rmsnorm_quant_ex(const void *x, const void *residual, const void *weight,
                                    float eps, int quant_mode, const float *scale_in,
                                    void *out_q, void *out_scales, void *residual_out,
                                    int64_t n_tokens, int64_t hidden, int dtype, void *stream,
                                    int variant);

/*
 * rmsq_fused_add_rmsnorm_nvfp4_dynamic — the NVFP4 mode with the global scale
 * taken from the data instead of scale_in: gs = 448 * 6 / amax(|y|) over the
 * whole batch (the NVFP4 workload's definition of the global scale; gs = 1
 * when that amax is 0), then exactly the RMSQ_NVFP4 quantisation with that gs
 * (vLLM PR #51925 summary, "Motivation": residual update + RMSNorm, block
 * scales, FP4 values, fp32 global scale).  Two kernels: the first computes
 * the residual, and the per-row inv_rms and per-CTA maxima of |y| into
 * `workspace`; the second takes the batch amax from those maxima, re-reads h
 * (residual_out, or x without a residual) and quantises.
 *  out_global_scale  device, one fp32 (4-byte aligned): receives gs.
 *  workspace         device, 16-byte aligned, at least
 *                    rmsq_nvfp4_dynamic_workspace_bytes(n_tokens) bytes of
 *                    caller-owned scratch; its contents on entry do not
 *                    matter and are overwritten.  Two calls in flight at the
 *                    same time must not share one workspace.
 *  variant           an rmsq_variant for the first pass.
 * Every other argument as in rmsq_fused_add_rmsnorm_quant with quant_mode
 * RMSQ_NVFP4 (out_block_scales = its out_scales).  RMSQ_ERR_INVALID_ARG also
 * for a NULL or too small workspace; no output may overlap the workspace.
 */
int rmsq_fused_add_rmsnorm_nvfp4_dynamic(const void *x, const void *residual, const void *weight,
                                         float eps, void *out_q, void *out_block_scales,
                                         float *out_global_scale, void *residual_out,
                                         void *workspace, size_t workspace_bytes,
                                         int64_t n_tokens, int64_t hidden, int dtype, void *stream,
                                         int variant);

/* Bytes of workspace rmsq_fused_add_rmsnorm_nvfp4_dynamic needs for n_tokens
 * rows: 256 + 8 * n_tokens (one fp32 inverse RMS per row and at most one
 * fp32 partial maximum per row), rounded up to a multiple of 256 (0 for
 * n < 0). */
size_t rmsq_nvfp4_dynamic_workspace_bytes(int64_t n_tokens);

/* Largest batch rmsq_fused_add_rmsnorm_nvfp4_dynamic_noalloc accepts. */
#define RMSQ_NOALLOC_MAX_TOKENS 65536

/*
 * rmsq_fused_add_rmsnorm_nvfp4_dynamic_noalloc — rmsq_fused_add_rmsnorm_nvfp4_dynamic
 * without a caller workspace and without any device allocation.  The pages
 * have no counterpart to this entry point: it exists for callers that cannot
 * allocate device memory themselves — for instance a plugin inside an engine
 * that owns all device memory through its own pool and hands the plugin none,
 * or latency-critical code that must not call cudaMalloc because it can
 * synchronise the device.  The caller still passes every input and output.
 *
 * The workspace lives in a fixed device array inside the library (256 + 8 *
 * RMSQ_NOALLOC_MAX_TOKENS bytes, about 513 KiB), present on every device that
 * loads the library until the process exits.  n_tokens above
 * RMSQ_NOALLOC_MAX_TOKENS returns RMSQ_ERR_UNSUPPORTED_SHAPE (use the entry
 * point with a workspace for larger batches).  Every call looks up the
 * array's device address in the current device's context
 * (cudaGetSymbolAddress), so a reset of the device's primary context between
 * calls is followed; the first call on a device may load the library's device
 * code there: make that first call before any stream capture.  Every call on a
 * device shares the one array and leaves its contents behind; nothing in it
 * has to start at zero (every call writes what it reads).  Calls whose work overlaps on
 * the GPU (other streams, or other host threads) race on the array: order them.
 * Arguments, results and every other rule are those of
 * rmsq_fused_add_rmsnorm_nvfp4_dynamic; without a CUDA device it returns
 * RMSQ_ERR_NO_DEVICE.
 */
int rmsq_fused_add_rmsnorm_nvfp4_dynamic_noalloc(const void *x, const void *residual,
                                                 const void *weight, float eps, void *out_q,
                                                 void *out_block_scales, float *out_global_scale,
                                                 void *residual_out, int64_t n_tokens,
                                                 int64_t hidden, int dtype, void *stream,
                                                 int variant);

/*
 * The unfused two-op sequence the fused op replaces (vLLM docs "Fusion
 * torch.compile passes", fuse_norm_quant: fused_add_rms_norm / rms_norm
 * followed by the quantisation op), for comparison and for callers that need
 * the normalised activations themselves.
 *
 * rmsq_fused_add_rmsnorm — steps 1-4 of rmsq_fused_add_rmsnorm_quant (residual
 * add and write-back, RMSNorm with the same canonical sum), then y rounded to
 * the activation type (nearest even) into y_out: device [n_tokens, hidden],
 * same type as x, 16-byte aligned, overlapping no input or residual_out.
 * Arguments and errors otherwise as rmsq_fused_add_rmsnorm_quant.
 *
 * rmsq_quant — the quantisation step of rmsq_fused_add_rmsnorm_quant applied
 * to a [n_tokens, hidden] tensor y of the activation type (widened exactly to
 * fp32): every quant_mode and scale option, same outputs and layouts.
 * Running the two in sequence gives the unfused result, which differs from
 * the fused op's in that y is rounded to the activation type in between.
 */
int rmsq_fused_add_rmsnorm(const void *x, const void *residual, const void *weight, float eps,
                           void *y_out, void *residual_out, int64_t n_tokens, int64_t hidden, int dtype,
                           void *stream);
int rmsq_quant(const void *y, int quant_mode, const float *scale_in, void *out_q, void *out_scales,
               int64_t n_tokens, int64_t hidden, int dtype, void *stream);

/*
 * rmsq_qk_norm_rope — QK-norm + RoPE in one kernel (vLLM docs "Fusion
 * torch.compile passes", section "QK Norm + RoPE (enable_qk_norm_rope_fusion)":
 * split QKV, per-head RMSNorm of Q and K, rotary embedding), in place.
 *  qkv            device, T[n_tokens, (num_q_heads + 2 num_kv_heads) head_dim]:
 *                 per token the q heads, then the k heads, then the v heads;
 *                 16-byte aligned; updated in place (v heads untouched).
 *  positions      device, int64[n_tokens], 8-byte aligned: each token's position.
 *  cos_sin_cache  device, fp32[max_positions, head_dim], 16-byte aligned: at
 *                 row p, cos of the head_dim/2 angles then their sin.
 *  q_weight, k_weight  device, T[head_dim], 16-byte aligned: the norm weights.
 * Per q / k head: S = canonical pairwise sum of x^2 over the head,
 * inv = 1 / sqrt(S / head_dim + eps), y = (x * inv) * w in fp32 (the norm op's
 * steps); then with c_i, s_i from row positions[t] of the table, each pair
 * (a, b) becomes (a c - b s, b c + a s) (every product and sum rounded to
 * fp32 separately), rounded once to T.  is_neox = 1 pairs element i with
 * i + head_dim/2, 0 pairs 2i with 2i + 1 (GPT-J); angle index i either way.
 * A token whose position is outside [0, max_positions) is left unchanged.
 * head_dim 64, 128 or 256 (else RMSQ_ERR_UNSUPPORTED_SHAPE); eps finite,
 * >= 0; no input may overlap qkv.  Asynchronous on `stream`.
 */
int rmsq_qk_norm_rope(void *qkv, const int64_t *positions, const float *cos_sin_cache,
                      int64_t max_positions, const void *q_weight, const void *k_weight, float eps,
                      int64_t n_tokens, int num_q_heads, int num_kv_heads, int head_dim, int is_neox,
                      int dtype, void *stream);

/*
 * rmsq_qk_norm_rope_ex — rmsq_qk_norm_rope with an explicit rmsq_variant
 * (RMSQ_ERR_INVALID_ARG for any other value); bit-identical results either
 * way.  DIRECT: each warp loads its heads straight into registers (lowest
 * latency for a few tokens).  PIPELINED: persistent CTAs keep the q and k
 * heads and the cos / sin rows of several tokens in flight as bulk
 * asynchronous copies into shared memory; it needs two tokens' q and k heads
 * plus their cos / sin rows within the shared-memory ring (about 110 KB per
 * CTA) and runs as DIRECT where they do not fit.  AUTO: PIPELINED from eight
 * tokens per SM up.
 */
int rmsq_qk_norm_rope_ex(void *qkv, const int64_t *positions, const float *cos_sin_cache,
                         int64_t max_positions, const void *q_weight, const void *k_weight, float eps,
                         int64_t n_tokens, int num_q_heads, int num_kv_heads, int head_dim, int is_neox,
                         int dtype, void *stream, int variant);

/* Most ranks rmsq_allreduce_add_rmsnorm_quant sums. */
#define RMSQ_MAX_ALLREDUCE_RANKS 8

/*
 * rmsq_allreduce_add_rmsnorm_quant — the tensor-parallel all-reduce fused with
 * the residual add, RMSNorm and quantisation (vLLM docs "Fusion torch.compile
 * passes", section "AllReduce + RMSNorm (fuse_allreduce_rms)": all-reduce ->
 * RMSNorm (+ residual add) (-> FP8 static or NVFP4 quantisation), worth it at
 * small token counts).  One-shot, by loads: for every row the kernel reads
 * the row of each rank's partial sums, adds them in rank order in fp32 and
 * rounds the sum once to T:
 *   x = T(fp32(partials[0]) + fp32(partials[1]) + ... + fp32(partials[n_ranks-1]))
 * and then computes exactly rmsq_fused_add_rmsnorm_quant on that x (every
 * quant_mode and option; the same outputs and layouts).
 *  partials     HOST array of n_ranks (1 .. RMSQ_MAX_ALLREDUCE_RANKS) device
 *               pointers, each T[n_tokens, hidden], 16-byte aligned, that
 *               the current device can read: its own memory, or another
 *               GPU's memory mapped into this device's address space (CUDA
 *               IPC or peer access, set up by the caller; the library maps
 *               nothing).  The pointer values are copied at the call.
 *  Every other argument as in rmsq_fused_add_rmsnorm_quant (residual may be
 *  NULL; residual_out == residual is the in-place update).
 * Ordering: the kernel does not wait for other GPUs.  Every rank's partials
 * must be complete before the launch in `stream`'s order (for instance a
 * stream wait on an event each producer recorded, or a host barrier after
 * the producers synchronised); with peer buffers the caller also keeps them
 * alive and unmodified until the call completes.  Each rank that needs the
 * result calls this on its own device with the same partials (a one-shot
 * all-reduce), or on its own slice of rows (pointers and n_tokens of that
 * slice) followed by an all-gather of the outputs (a two-shot one).
 * No output may overlap a partial; RMSQ_ERR_INVALID_ARG for a NULL array or
 * pointer or a bad n_ranks.  Asynchronous on `stream`.
 */
int rmsq_allreduce_add_rmsnorm_quant(const void *const *partials, int n_ranks, const void *residual,
                                     const void *weight, float eps, int quant_mode,
                                     const float *scale_in, void *out_q, void *out_scales,
                                     void *residual_out, int64_t n_tokens, int64_t hidden,
                                     int dtype, void *stream);

/* Largest d (activation width) of rmsq_silu_mul_quant. */
#define RMSQ_ACT_MAX_D 32768

/*
 * rmsq_silu_mul_quant — SiLU+Mul + activation quantisation in one kernel (vLLM
 * docs "Fusion torch.compile passes", section "SiLU+Mul + Quantization
 * (fuse_act_quant)": silu_and_mul on the gated up-projection followed by the
 * quantisation, without the full-precision activation tensor in between).
 * Per row t: a_i = silu(g_i) * u_i in fp32, silu(g) = g / (1 + e^-g) with
 * g_i = gate_up[t, i] and u_i = gate_up[t, d + i]; then exactly the
 * quantisation step of rmsq_fused_add_rmsnorm_quant with a in place of y
 * (every quant_mode; scales and codes laid out the same way with hidden = d).
 * e^x follows W. J. Cody and W. Waite's argument reduction, then the
 * hardware's approximate 2^x on the reduced argument (within about 2.4 ulp
 * of e^x over the normal range); the quotient is g times the hardware's
 * approximate reciprocal of 1 + e^-g (within one ulp), so a is within
 * 9.8 * 2^-24 relative of the exact silu(g) * u (results are deterministic:
 * the same inputs always give the same bytes).  Where e^-g
 * overflows (g < -88.72) silu is -0.  The quantisation of a is exact, as in
 * the norm op.
 *  gate_up     device, [n_tokens, 2 d] bf16/fp16, row-major, 16-byte aligned.
 *  quant_mode  an rmsq_quant_mode, optionally OR-ed with RMSQ_QUANT_* options.
 *  scale_in    device fp32: FP8 static scale or NVFP4 global scale (else
 *              ignored, may be NULL).
 *  out_q       device: [n, d] E4M3 bytes, or [n, d/2] E2M1 pairs for NVFP4.
 *  out_scales  device: as for rmsq_fused_add_rmsnorm_quant with hidden = d.
 *  n_tokens    >= 0 (0 returns RMSQ_OK without a launch);
 *  d           > 0, a multiple of 8 (16 for NVFP4, the group for group
 *              modes), at most RMSQ_ACT_MAX_D (else
 *              RMSQ_ERR_UNSUPPORTED_SHAPE).
 * Errors as for rmsq_fused_add_rmsnorm_quant (no output may overlap an input
 * or another output).  Asynchronous on `stream`; the caller owns all memory.
 */
int rmsq_silu_mul_quant(const void *gate_up, int quant_mode, const float *scale_in, void *out_q,
                        void *out_scales, int64_t n_tokens, int64_t d, int dtype, void *stream);

/*
 * rmsq_set_pipeline_config — process-wide tuning of the PIPELINED variant:
 * chunks_per_thread (16-byte chunks of a row per thread: 1, 2, 4 or 8),
 * stages (rows in flight per CTA: 1..8) and ctas_per_sm (cap on resident
 * CTAs per SM: 1..32).  rows_per_iter (0, 1 or 2) is accepted and has no
 * effect: the norm kernels work on one row per CTA iteration.  0 keeps the
 * automatic choice for that parameter.  The pipelined QK-norm + RoPE kernel takes stages (tokens
 * in flight per CTA, 2..8) and ctas_per_sm from the same settings.  A choice
 * that does not fit (more than 512 threads, or a ring larger than the shared
 * memory budget) falls back to the automatic one.  Results do not depend on
 * these settings.  Not synchronised with launches running concurrently on
 * other host threads.
 */
int rmsq_set_pipeline_config(int chunks_per_thread, int stages, int ctas_per_sm, int rows_per_iter);

/*
 * rmsq_set_programmatic_launch — process-wide: 1 (the default) launches every
 * kernel with programmatic stream serialisation (programmatic dependent
 * launch), 0 with plain stream order.  With it, a kernel may be scheduled
 * while the previous kernel in the stream is still finishing, which hides the
 * launch gap between back-to-back calls (in a CUDA graph as well); each
 * kernel still waits for the previous one to complete, with its memory
 * visible, before its first global memory access, so stream semantics and
 * results are unchanged.  The pages have no counterpart: it is a launch
 * detail of this implementation.  Returns RMSQ_ERR_INVALID_ARG for a value
 * other than 0 or 1.  Not synchronised with launches on other host threads.
 */
int rmsq_set_programmatic_launch(int enable);

/*
 * rmsq_take_fault_flags — reads and clears, on the current device, the flag a
 * pipelined launch (norm or QK-norm + RoPE) sets if it ever gives up
 * waiting (after 100 ms) for its own shared-memory copies; the outputs of
 * such a launch are incomplete.
 * *flags = 0 when no launch gave up.  Synchronous with respect to the device:
 * call it after the launches of interest have completed.
 */
int rmsq_take_fault_flags(uint32_t *flags);

/*
 * rmsq_query_sizes — bytes of out_q and out_scales for a mode and shape (host
 * only, no device needed).  scale_bytes is 0 for FP8_STATIC.
 */
int rmsq_query_sizes(int quant_mode, int64_t n_tokens, int64_t hidden, size_t *q_bytes,
                     size_t *scale_bytes);

/*
 * rmsq_query_launch — the launch rmsq_fused_add_rmsnorm_quant_ex would make on
 * the current device for a mode, shape, residual (0/1), dtype and variant,
 * without launching anything: out[0] = 1 for the pipelined kernel, 0 for the
 * direct one; out[1] = 16-byte chunks per thread; out[2] = ring stages (0
 * for the direct kernel); out[3] = CTAs; out[4] = threads per CTA (all 0 for
 * n_tokens = 0).  The pages have no counterpart: it reports this
 * implementation's choice (for profiling and tuning).  out: host, 5 int32.
 * Errors as for rmsq_fused_add_rmsnorm_quant_ex's mode, shape, dtype and
 * variant; RMSQ_ERR_NO_DEVICE / RMSQ_ERR_UNSUPPORTED_DEVICE without a
 * suitable device.
 */
int rmsq_query_launch(int quant_mode, int64_t n_tokens, int64_t hidden, int has_residual, int dtype,
                      int variant, int32_t *out);

/*
 * rmsq_debug_convert — the library's own fp32 -> 8-bit / 4-bit conversions on
 * a device array, so that tests can pin them against a reference encoder.
 * kind 0: out[i] = e4m3(in[i]) (E4M3FN, nearest even, saturating);
 * kind 1: out[i] = e2m1(in[i]) in the low nibble (high nibble 0).
 * in: device fp32[n]; out: device u8[n]; no alignment requirement.
 */
int rmsq_debug_convert(int kind, const float *in, uint8_t *out, int64_t n, void *stream);

/*
 * rmsq_debug_activation — the library's own e^x and SiLU steps (those of
 * rmsq_silu_mul_quant) on device arrays, so that tests can compare them with
 * a reference element by element.  kind 0: out[i] = e^in[i]; kind 1:
 * out[i] = silu(in[i]); kind 2: out[i] = silu(in[i]) * in2[i] (in2 is
 * ignored otherwise and may be NULL); kind 3: e^in[i] by the shorter steps
 * the kernel takes when |in[i]| <= 87 (defined only there).  Device fp32 arrays of n elements,
 * 4-byte aligned; out must not overlap the inputs.
 */
int rmsq_debug_activation(int kind, const float *in, const float *in2, float *out, int64_t n,
                          void *stream);

/*
 * rmsq_debug_bounded_wait — failure detection without a fault: one CTA waits
 * on a shared-memory barrier that nothing ever completes, with the same
 * bounded wait the pipelined kernels use on their copies, here limited to
 * limit_ns (1 .. 1e9).  *gave_up = 1 when every thread gave up and the kernel
 * returned normally (the expected outcome), 0 if none did, 2 if only some
 * did.  Synchronous (waits for the device); the context stays usable.
 */
int rmsq_debug_bounded_wait(int64_t limit_ns, int *gave_up);

/* Text for an rmsq_status (static storage, never NULL). */
const char *rmsq_status_string(int status);

/* CUDA error code (cudaError_t) of the last RMSQ_ERR_CUDA on this thread. */
int rmsq_last_cuda_error(void);

/* RMSQ_VERSION of the built library. */
int rmsq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RMSQ_H */

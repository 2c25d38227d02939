// C ABI of librmsq: argument checks, device check, dispatch.  Declarations and
// the meaning of every argument are in include/rmsq.h.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "rmsq.h"
#include "rmsq_abi.h"
#include "rmsq_launch.h"

namespace {

thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 128;
// Per-device compute capability (major * 10 + minor), 0 = not yet queried.
std::atomic<int> g_cc[kMaxDevices];
// Device count: -1 = not yet queried.
std::atomic<int> g_device_count{-1};

}  // namespace

namespace rmsq_abi {

int fail_cuda(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();   // a non-sticky error is not left pending for later calls
    return RMSQ_ERR_CUDA;
}

// RMSQ_OK when the current device is a compute capability 10.3 part.
int check_device() {
    int count = g_device_count.load(std::memory_order_acquire);
    if (count < 0) {
        cudaError_t e = cudaGetDeviceCount(&count);
        if (e != cudaSuccess) {
            cudaGetLastError();
            count = 0;
        }
        g_device_count.store(count, std::memory_order_release);
    }
    if (count == 0) return RMSQ_ERR_NO_DEVICE;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return RMSQ_ERR_UNSUPPORTED_DEVICE;
    int cc = g_cc[dev].load(std::memory_order_acquire);
    if (cc == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return fail_cuda(e);
        cc = major * 10 + minor;
        g_cc[dev].store(cc, std::memory_order_release);
    }
    return cc == 103 ? RMSQ_OK : RMSQ_ERR_UNSUPPORTED_DEVICE;
}

}  // namespace rmsq_abi

namespace {

using rmsq_abi::check_device;
using rmsq_abi::fail_cuda;

int group_of(int mode) {
    switch (mode) {
    case RMSQ_FP8_GROUP128_ROW:
    case RMSQ_FP8_GROUP128_COL: return 128;
    case RMSQ_FP8_GROUP64_ROW:
    case RMSQ_FP8_GROUP64_COL: return 64;
    default: return 0;
    }
}

// Option bits of a quant_mode argument: only with a dynamic FP8 scale
// (E8M0) or with column-major group scales (TMA-aligned stride).
bool options_valid(int quant_mode) {
    const int base = quant_mode & RMSQ_QUANT_MODE_MASK, opts = quant_mode & ~RMSQ_QUANT_MODE_MASK;
    if (opts & ~(RMSQ_QUANT_E8M0 | RMSQ_QUANT_TMA_ALIGNED | RMSQ_QUANT_UE8M0)) return false;
    const bool dynamic = base >= RMSQ_FP8_PER_TOKEN && base <= RMSQ_FP8_GROUP64_COL;
    const bool col = base == RMSQ_FP8_GROUP128_COL || base == RMSQ_FP8_GROUP64_COL;
    return !((opts & (RMSQ_QUANT_E8M0 | RMSQ_QUANT_UE8M0)) && !dynamic) &&
           !((opts & RMSQ_QUANT_TMA_ALIGNED) && !col);
}

// Bytes per dynamic FP8 scale: 4 (fp32), 1 with the UE8M0 byte option.
int scale_elem_bytes(int quant_mode) { return (quant_mode & RMSQ_QUANT_UE8M0) ? 1 : 4; }

// Column-major stride: n, or n rounded up to 16 bytes of scales.
int64_t col_stride_of(int quant_mode, int64_t n) {
    const int64_t per16 = 16 / scale_elem_bytes(quant_mode);
    return (quant_mode & RMSQ_QUANT_TMA_ALIGNED) ? (n + per16 - 1) / per16 * per16 : n;
}

int check_shape(int quant_mode, int64_t n, int64_t hidden) {
    if (quant_mode < 0 || !options_valid(quant_mode)) return RMSQ_ERR_INVALID_ARG;
    const int mode = quant_mode & RMSQ_QUANT_MODE_MASK;
    if (mode < RMSQ_FP8_STATIC || mode > RMSQ_NVFP4) return RMSQ_ERR_INVALID_ARG;
    if (n < 0 || hidden <= 0) return RMSQ_ERR_INVALID_ARG;
    if (n > INT32_MAX || hidden > RMSQ_MAX_HIDDEN || hidden % 8 != 0) return RMSQ_ERR_UNSUPPORTED_SHAPE;
    if (mode == RMSQ_NVFP4 && hidden % 16 != 0) return RMSQ_ERR_UNSUPPORTED_SHAPE;
    const int g = group_of(mode);
    if (g && hidden % g != 0) return RMSQ_ERR_UNSUPPORTED_SHAPE;
    return RMSQ_OK;
}

void sizes_of(int quant_mode, int64_t n, int64_t hidden, size_t* q, size_t* sc) {
    const int mode = quant_mode & RMSQ_QUANT_MODE_MASK;
    *q = static_cast<size_t>(mode == RMSQ_NVFP4 ? n * (hidden / 2) : n * hidden);
    switch (mode) {
    case RMSQ_FP8_STATIC: *sc = 0; break;
    case RMSQ_FP8_PER_TOKEN: *sc = static_cast<size_t>(n) * scale_elem_bytes(quant_mode); break;
    case RMSQ_NVFP4: *sc = static_cast<size_t>(n * (hidden / 16)); break;
    case RMSQ_FP8_GROUP128_COL:
    case RMSQ_FP8_GROUP64_COL:
        *sc = static_cast<size_t>(col_stride_of(quant_mode, n) * (hidden / group_of(mode))) *
              scale_elem_bytes(quant_mode);
        break;
    default: *sc = static_cast<size_t>(n * (hidden / group_of(mode))) * scale_elem_bytes(quant_mode); break;
    }
}

struct Span {
    uintptr_t lo, hi;   // [lo, hi); empty when lo == hi
};

Span span(const void* p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, p ? a + bytes : a};
}

bool overlaps(Span a, Span b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

std::atomic<int> g_tune_j{0}, g_tune_stages{0}, g_tune_cps{0}, g_tune_rows{0};
std::atomic<bool> g_pdl{true};

}  // namespace

namespace rmsq {
PipeTuning get_pipe_tuning() {
    return {g_tune_j.load(std::memory_order_relaxed), g_tune_stages.load(std::memory_order_relaxed),
            g_tune_cps.load(std::memory_order_relaxed), g_tune_rows.load(std::memory_order_relaxed)};
}
void set_pipe_tuning(const PipeTuning& t) {
    g_tune_j.store(t.chunks_per_thread, std::memory_order_relaxed);
    g_tune_stages.store(t.stages, std::memory_order_relaxed);
    g_tune_cps.store(t.ctas_per_sm, std::memory_order_relaxed);
    g_tune_rows.store(t.rows_per_iter, std::memory_order_relaxed);
}
bool programmatic_launch() { return g_pdl.load(std::memory_order_relaxed); }
void set_programmatic_launch(bool on) { g_pdl.store(on, std::memory_order_relaxed); }
}  // namespace rmsq

extern "C" {

int rmsq_set_pipeline_config(int chunks_per_thread, int stages, int ctas_per_sm, int rows_per_iter) {
    if (chunks_per_thread != 0 && chunks_per_thread != 1 && chunks_per_thread != 2 && chunks_per_thread != 4 &&
        chunks_per_thread != 8)
        return RMSQ_ERR_INVALID_ARG;
    if (stages < 0 || stages > 8 || ctas_per_sm < 0 || ctas_per_sm > 32) return RMSQ_ERR_INVALID_ARG;
    if (rows_per_iter < 0 || rows_per_iter > 2) return RMSQ_ERR_INVALID_ARG;
    rmsq::set_pipe_tuning({chunks_per_thread, stages, ctas_per_sm, rows_per_iter});
    return RMSQ_OK;
}

int rmsq_set_programmatic_launch(int enable) {
    if (enable != 0 && enable != 1) return RMSQ_ERR_INVALID_ARG;
    rmsq::set_programmatic_launch(enable == 1);
    return RMSQ_OK;
}

int rmsq_fused_add_rmsnorm_quant_ex(const void* x, const void* residual, const void* weight, float eps,
                                    int quant_mode, const float* scale_in, void* out_q, void* out_scales,
                                    void* residual_out, int64_t n_tokens, int64_t hidden, int dtype,
                                    void* stream, int variant) {
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    if (variant != RMSQ_VARIANT_AUTO && variant != RMSQ_VARIANT_DIRECT && variant != RMSQ_VARIANT_PIPELINED)
        return RMSQ_ERR_INVALID_ARG;
    int st = check_shape(quant_mode, n_tokens, hidden);
    if (st != RMSQ_OK) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSQ_ERR_INVALID_ARG;
    if (n_tokens == 0) return RMSQ_OK;
    const int mode = quant_mode & RMSQ_QUANT_MODE_MASK;

    const bool needs_scale_in = mode == RMSQ_FP8_STATIC || mode == RMSQ_NVFP4;
    const bool has_scales = mode != RMSQ_FP8_STATIC;
    if (!x || !weight || !out_q) return RMSQ_ERR_INVALID_ARG;
    if ((residual == nullptr) != (residual_out == nullptr)) return RMSQ_ERR_INVALID_ARG;
    if (needs_scale_in && !scale_in) return RMSQ_ERR_INVALID_ARG;
    if (has_scales && !out_scales) return RMSQ_ERR_INVALID_ARG;
    if (!needs_scale_in) scale_in = nullptr;
    if (!has_scales) out_scales = nullptr;

    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(weight, 16) ||
        !aligned(residual_out, 16) || !aligned(out_q, 16) || !aligned(scale_in, 4))
        return RMSQ_ERR_ALIGNMENT;
    if (mode != RMSQ_NVFP4 && !aligned(out_scales, scale_elem_bytes(quant_mode))) return RMSQ_ERR_ALIGNMENT;

    size_t q_bytes = 0, sc_bytes = 0;
    sizes_of(quant_mode, n_tokens, hidden, &q_bytes, &sc_bytes);
    const size_t act = static_cast<size_t>(n_tokens * hidden) * 2;
    const Span X = span(x, act), R = span(residual, act), W = span(weight, hidden * 2),
               RO = span(residual_out, act), Q = span(out_q, q_bytes), SC = span(out_scales, sc_bytes),
               SI = span(scale_in, 4);
    if (residual && X.lo != R.lo && overlaps(X, R)) return RMSQ_ERR_ALIAS;
    if (residual_out) {
        if (RO.lo != X.lo && overlaps(RO, X)) return RMSQ_ERR_ALIAS;
        if (RO.lo != R.lo && overlaps(RO, R)) return RMSQ_ERR_ALIAS;
        if (overlaps(RO, W) || overlaps(RO, SI)) return RMSQ_ERR_ALIAS;
    }
    const Span outs[2] = {Q, SC};
    for (const Span& o : outs)
        if (overlaps(o, X) || overlaps(o, R) || overlaps(o, W) || overlaps(o, RO) || overlaps(o, SI))
            return RMSQ_ERR_ALIAS;
    if (overlaps(Q, SC)) return RMSQ_ERR_ALIAS;

    st = check_device();
    if (st != RMSQ_OK) return st;

    rmsq::LaunchArgs la = {};
    la.x = x;
    la.res = residual;
    la.w = weight;
    la.res_out = residual_out;
    la.q = out_q;
    la.scales = out_scales;
    la.scale_in = scale_in;
    la.eps = eps;
    la.mode = mode;
    la.e8m0 = (quant_mode & (RMSQ_QUANT_E8M0 | RMSQ_QUANT_UE8M0)) != 0;
    la.ue8m0 = (quant_mode & RMSQ_QUANT_UE8M0) != 0;
    la.col_stride = static_cast<int>(col_stride_of(quant_mode, n_tokens));
    la.n = static_cast<int>(n_tokens);
    la.hidden = static_cast<int>(hidden);
    la.variant = variant == RMSQ_VARIANT_DIRECT ? rmsq::kVariantDirect
                 : variant == RMSQ_VARIANT_PIPELINED ? rmsq::kVariantPipelined : rmsq::kVariantAuto;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == RMSQ_BF16 ? rmsq::launch_rows_bf16(la, s) : rmsq::launch_rows_fp16(la, s);
    if (e != cudaSuccess) return fail_cuda(e);
    return RMSQ_OK;
}

int rmsq_query_launch(int quant_mode, int64_t n_tokens, int64_t hidden, int has_residual, int dtype, int variant,
                      int32_t* out) {
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    if (variant != RMSQ_VARIANT_AUTO && variant != RMSQ_VARIANT_DIRECT && variant != RMSQ_VARIANT_PIPELINED)
        return RMSQ_ERR_INVALID_ARG;
    if ((has_residual != 0 && has_residual != 1) || !out) return RMSQ_ERR_INVALID_ARG;
    int st = check_shape(quant_mode, n_tokens, hidden);
    if (st != RMSQ_OK) return st;
    if (n_tokens == 0) {
        for (int i = 0; i < 5; ++i) out[i] = 0;
        return RMSQ_OK;
    }
    st = check_device();
    if (st != RMSQ_OK) return st;
    // Only the shape matters for the plan; the pointers stand for aligned
    // buffers (the direct kernel's paired accesses take them when they are).
    alignas(32) static unsigned char dummy[32];
    rmsq::LaunchArgs la = {};
    la.x = dummy;
    la.res = has_residual ? dummy : nullptr;
    la.w = dummy;
    la.res_out = has_residual ? dummy : nullptr;
    la.mode = quant_mode & RMSQ_QUANT_MODE_MASK;
    la.n = static_cast<int>(n_tokens);
    la.hidden = static_cast<int>(hidden);
    la.variant = variant == RMSQ_VARIANT_DIRECT ? rmsq::kVariantDirect
                 : variant == RMSQ_VARIANT_PIPELINED ? rmsq::kVariantPipelined : rmsq::kVariantAuto;
    int v[5] = {0, 0, 0, 0, 0};
    const cudaError_t e = dtype == RMSQ_BF16 ? rmsq::query_rows_bf16(la, v) : rmsq::query_rows_fp16(la, v);
    if (e != cudaSuccess) return fail_cuda(e);
    for (int i = 0; i < 5; ++i) out[i] = v[i];
    return RMSQ_OK;
}

int rmsq_allreduce_add_rmsnorm_quant(const void* const* partials, int n_ranks, const void* residual,
                                     const void* weight, float eps, int quant_mode, const float* scale_in,
                                     void* out_q, void* out_scales, void* residual_out, int64_t n_tokens,
                                     int64_t hidden, int dtype, void* stream) {
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    if (!partials || n_ranks < 1 || n_ranks > RMSQ_MAX_ALLREDUCE_RANKS) return RMSQ_ERR_INVALID_ARG;
    int st = check_shape(quant_mode, n_tokens, hidden);
    if (st != RMSQ_OK) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSQ_ERR_INVALID_ARG;
    if (n_tokens == 0) return RMSQ_OK;
    const int mode = quant_mode & RMSQ_QUANT_MODE_MASK;
    const bool needs_scale_in = mode == RMSQ_FP8_STATIC || mode == RMSQ_NVFP4;
    const bool has_scales = mode != RMSQ_FP8_STATIC;
    if (!weight || !out_q) return RMSQ_ERR_INVALID_ARG;
    for (int r = 0; r < n_ranks; ++r)
        if (!partials[r]) return RMSQ_ERR_INVALID_ARG;
    if ((residual == nullptr) != (residual_out == nullptr)) return RMSQ_ERR_INVALID_ARG;
    if (needs_scale_in && !scale_in) return RMSQ_ERR_INVALID_ARG;
    if (has_scales && !out_scales) return RMSQ_ERR_INVALID_ARG;
    if (!needs_scale_in) scale_in = nullptr;
    if (!has_scales) out_scales = nullptr;
    for (int r = 0; r < n_ranks; ++r)
        if (!aligned(partials[r], 16)) return RMSQ_ERR_ALIGNMENT;
    if (!aligned(residual, 16) || !aligned(weight, 16) || !aligned(residual_out, 16) || !aligned(out_q, 16) ||
        !aligned(scale_in, 4))
        return RMSQ_ERR_ALIGNMENT;
    if (mode != RMSQ_NVFP4 && !aligned(out_scales, scale_elem_bytes(quant_mode))) return RMSQ_ERR_ALIGNMENT;

    size_t q_bytes = 0, sc_bytes = 0;
    sizes_of(quant_mode, n_tokens, hidden, &q_bytes, &sc_bytes);
    const size_t act = static_cast<size_t>(n_tokens * hidden) * 2;
    const Span R = span(residual, act), W = span(weight, hidden * 2), RO = span(residual_out, act),
               Q = span(out_q, q_bytes), SC = span(out_scales, sc_bytes), SI = span(scale_in, 4);
    const Span outs[3] = {RO, Q, SC};
    for (int r = 0; r < n_ranks; ++r) {
        const Span P = span(partials[r], act);
        for (const Span& o : outs)
            if (overlaps(o, P)) return RMSQ_ERR_ALIAS;
    }
    if (residual_out) {
        if (RO.lo != R.lo && overlaps(RO, R)) return RMSQ_ERR_ALIAS;
        if (overlaps(RO, W) || overlaps(RO, SI)) return RMSQ_ERR_ALIAS;
    }
    const Span qs[2] = {Q, SC};
    for (const Span& o : qs)
        if (overlaps(o, R) || overlaps(o, W) || overlaps(o, RO) || overlaps(o, SI)) return RMSQ_ERR_ALIAS;
    if (overlaps(Q, SC)) return RMSQ_ERR_ALIAS;

    st = check_device();
    if (st != RMSQ_OK) return st;
    rmsq::LaunchArgs la = {};
    la.res = residual;
    la.w = weight;
    la.res_out = residual_out;
    la.q = out_q;
    la.scales = out_scales;
    la.scale_in = scale_in;
    la.eps = eps;
    la.mode = mode;
    la.e8m0 = (quant_mode & (RMSQ_QUANT_E8M0 | RMSQ_QUANT_UE8M0)) != 0;
    la.ue8m0 = (quant_mode & RMSQ_QUANT_UE8M0) != 0;
    la.col_stride = static_cast<int>(col_stride_of(quant_mode, n_tokens));
    la.n = static_cast<int>(n_tokens);
    la.hidden = static_cast<int>(hidden);
    la.variant = rmsq::kVariantDirect;
    const cudaError_t e = rmsq::launch_allreduce_rows(la, partials, n_ranks, dtype == RMSQ_FP16,
                                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RMSQ_OK : fail_cuda(e);
}

int rmsq_silu_mul_quant(const void* gate_up, int quant_mode, const float* scale_in, void* out_q,
                        void* out_scales, int64_t n_tokens, int64_t d, int dtype, void* stream) {
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    if (quant_mode < 0 || !options_valid(quant_mode)) return RMSQ_ERR_INVALID_ARG;
    const int mode = quant_mode & RMSQ_QUANT_MODE_MASK;
    if (mode < RMSQ_FP8_STATIC || mode > RMSQ_NVFP4) return RMSQ_ERR_INVALID_ARG;
    if (n_tokens < 0 || d <= 0) return RMSQ_ERR_INVALID_ARG;
    if (n_tokens > INT32_MAX || d > RMSQ_ACT_MAX_D) return RMSQ_ERR_UNSUPPORTED_SHAPE;
    int st = check_shape(quant_mode, n_tokens, d <= RMSQ_MAX_HIDDEN ? d : 8);
    if (st != RMSQ_OK) return st;
    if (d % 8 != 0 || (mode == RMSQ_NVFP4 && d % 16 != 0) || (group_of(mode) && d % group_of(mode) != 0))
        return RMSQ_ERR_UNSUPPORTED_SHAPE;
    if (n_tokens == 0) return RMSQ_OK;

    const bool needs_scale_in = mode == RMSQ_FP8_STATIC || mode == RMSQ_NVFP4;
    const bool has_scales = mode != RMSQ_FP8_STATIC;
    if (!gate_up || !out_q) return RMSQ_ERR_INVALID_ARG;
    if (needs_scale_in && !scale_in) return RMSQ_ERR_INVALID_ARG;
    if (has_scales && !out_scales) return RMSQ_ERR_INVALID_ARG;
    if (!needs_scale_in) scale_in = nullptr;
    if (!has_scales) out_scales = nullptr;
    if (!aligned(gate_up, 16) || !aligned(out_q, 16) || !aligned(scale_in, 4)) return RMSQ_ERR_ALIGNMENT;
    if (mode != RMSQ_NVFP4 && !aligned(out_scales, scale_elem_bytes(quant_mode))) return RMSQ_ERR_ALIGNMENT;

    size_t q_bytes = 0, sc_bytes = 0;
    sizes_of(quant_mode, n_tokens, d, &q_bytes, &sc_bytes);
    const Span GU = span(gate_up, static_cast<size_t>(n_tokens * d) * 4), Q = span(out_q, q_bytes),
               SC = span(out_scales, sc_bytes), SI = span(scale_in, 4);
    const Span outs[2] = {Q, SC};
    for (const Span& o : outs)
        if (overlaps(o, GU) || overlaps(o, SI)) return RMSQ_ERR_ALIAS;
    if (overlaps(Q, SC)) return RMSQ_ERR_ALIAS;

    st = check_device();
    if (st != RMSQ_OK) return st;

    rmsq::LaunchArgs la = {};
    la.x = gate_up;
    la.q = out_q;
    la.scales = out_scales;
    la.scale_in = scale_in;
    la.mode = mode;
    la.e8m0 = (quant_mode & (RMSQ_QUANT_E8M0 | RMSQ_QUANT_UE8M0)) != 0;
    la.ue8m0 = (quant_mode & RMSQ_QUANT_UE8M0) != 0;
    la.col_stride = static_cast<int>(col_stride_of(quant_mode, n_tokens));
    la.n = static_cast<int>(n_tokens);
    la.hidden = static_cast<int>(d);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == RMSQ_BF16 ? rmsq::launch_act_bf16(la, s) : rmsq::launch_act_fp16(la, s);
    if (e != cudaSuccess) return fail_cuda(e);
    return RMSQ_OK;
}

int rmsq_fused_add_rmsnorm(const void* x, const void* residual, const void* weight, float eps, void* y_out,
                           void* residual_out, int64_t n_tokens, int64_t hidden, int dtype, void* stream) {
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    int st = check_shape(RMSQ_FP8_STATIC, n_tokens, hidden);
    if (st != RMSQ_OK) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSQ_ERR_INVALID_ARG;
    if (n_tokens == 0) return RMSQ_OK;
    if (!x || !weight || !y_out) return RMSQ_ERR_INVALID_ARG;
    if ((residual == nullptr) != (residual_out == nullptr)) return RMSQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(weight, 16) || !aligned(residual_out, 16) ||
        !aligned(y_out, 16))
        return RMSQ_ERR_ALIGNMENT;
    const size_t act = static_cast<size_t>(n_tokens * hidden) * 2;
    const Span X = span(x, act), R = span(residual, act), W = span(weight, hidden * 2),
               RO = span(residual_out, act), Y = span(y_out, act);
    if (residual && X.lo != R.lo && overlaps(X, R)) return RMSQ_ERR_ALIAS;
    if (residual_out) {
        if (RO.lo != X.lo && overlaps(RO, X)) return RMSQ_ERR_ALIAS;
        if (RO.lo != R.lo && overlaps(RO, R)) return RMSQ_ERR_ALIAS;
        if (overlaps(RO, W)) return RMSQ_ERR_ALIAS;
    }
    if (overlaps(Y, X) || overlaps(Y, R) || overlaps(Y, W) || overlaps(Y, RO)) return RMSQ_ERR_ALIAS;
    st = check_device();
    if (st != RMSQ_OK) return st;

    rmsq::LaunchArgs la = {};
    la.x = x;
    la.res = residual;
    la.w = weight;
    la.res_out = residual_out;
    la.q = y_out;
    la.eps = eps;
    la.mode = rmsq::kModeNormOnly;
    la.col_stride = static_cast<int>(n_tokens);
    la.n = static_cast<int>(n_tokens);
    la.hidden = static_cast<int>(hidden);
    la.variant = rmsq::kVariantAuto;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == RMSQ_BF16 ? rmsq::launch_rows_bf16(la, s) : rmsq::launch_rows_fp16(la, s);
    if (e != cudaSuccess) return fail_cuda(e);
    return RMSQ_OK;
}

int rmsq_quant(const void* y, int quant_mode, const float* scale_in, void* out_q, void* out_scales,
               int64_t n_tokens, int64_t hidden, int dtype, void* stream) {
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    int st = check_shape(quant_mode, n_tokens, hidden);
    if (st != RMSQ_OK) return st;
    if (n_tokens == 0) return RMSQ_OK;
    const int mode = quant_mode & RMSQ_QUANT_MODE_MASK;
    const bool needs_scale_in = mode == RMSQ_FP8_STATIC || mode == RMSQ_NVFP4;
    const bool has_scales = mode != RMSQ_FP8_STATIC;
    if (!y || !out_q) return RMSQ_ERR_INVALID_ARG;
    if (needs_scale_in && !scale_in) return RMSQ_ERR_INVALID_ARG;
    if (has_scales && !out_scales) return RMSQ_ERR_INVALID_ARG;
    if (!needs_scale_in) scale_in = nullptr;
    if (!has_scales) out_scales = nullptr;
    if (!aligned(y, 16) || !aligned(out_q, 16) || !aligned(scale_in, 4)) return RMSQ_ERR_ALIGNMENT;
    if (mode != RMSQ_NVFP4 && !aligned(out_scales, scale_elem_bytes(quant_mode))) return RMSQ_ERR_ALIGNMENT;
    size_t q_bytes = 0, sc_bytes = 0;
    sizes_of(quant_mode, n_tokens, hidden, &q_bytes, &sc_bytes);
    const Span Yi = span(y, static_cast<size_t>(n_tokens * hidden) * 2), Q = span(out_q, q_bytes),
               SC = span(out_scales, sc_bytes), SI = span(scale_in, 4);
    const Span outs[2] = {Q, SC};
    for (const Span& o : outs)
        if (overlaps(o, Yi) || overlaps(o, SI)) return RMSQ_ERR_ALIAS;
    if (overlaps(Q, SC)) return RMSQ_ERR_ALIAS;
    st = check_device();
    if (st != RMSQ_OK) return st;

    rmsq::LaunchArgs la = {};
    la.x = y;
    la.q = out_q;
    la.scales = out_scales;
    la.scale_in = scale_in;
    la.mode = mode;
    la.e8m0 = (quant_mode & (RMSQ_QUANT_E8M0 | RMSQ_QUANT_UE8M0)) != 0;
    la.ue8m0 = (quant_mode & RMSQ_QUANT_UE8M0) != 0;
    la.col_stride = static_cast<int>(col_stride_of(quant_mode, n_tokens));
    la.n = static_cast<int>(n_tokens);
    la.hidden = static_cast<int>(hidden);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == RMSQ_BF16 ? rmsq::launch_quant_bf16(la, s) : rmsq::launch_quant_fp16(la, s);
    if (e != cudaSuccess) return fail_cuda(e);
    return RMSQ_OK;
}

int rmsq_qk_norm_rope_ex(void* qkv, const int64_t* positions, const float* cos_sin_cache, int64_t max_positions,
                         const void* q_weight, const void* k_weight, float eps, int64_t n_tokens, int num_q_heads,
                         int num_kv_heads, int head_dim, int is_neox, int dtype, void* stream, int variant) {
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    if (variant != RMSQ_VARIANT_AUTO && variant != RMSQ_VARIANT_DIRECT && variant != RMSQ_VARIANT_PIPELINED)
        return RMSQ_ERR_INVALID_ARG;
    if (n_tokens < 0 || num_q_heads < 0 || num_kv_heads < 0 || num_q_heads + num_kv_heads == 0 ||
        max_positions <= 0 || (is_neox != 0 && is_neox != 1))
        return RMSQ_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSQ_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return RMSQ_ERR_UNSUPPORTED_SHAPE;
    if (num_q_heads > 4096 || num_kv_heads > 4096 ||
        n_tokens * (num_q_heads + num_kv_heads) > static_cast<int64_t>(INT32_MAX))
        return RMSQ_ERR_UNSUPPORTED_SHAPE;
    if (n_tokens == 0) return RMSQ_OK;
    if (!qkv || !positions || !cos_sin_cache || !q_weight || !k_weight) return RMSQ_ERR_INVALID_ARG;
    if (!aligned(qkv, 16) || !aligned(positions, 8) || !aligned(cos_sin_cache, 16) || !aligned(q_weight, 16) ||
        !aligned(k_weight, 16))
        return RMSQ_ERR_ALIGNMENT;
    const int64_t width = static_cast<int64_t>(num_q_heads + 2 * num_kv_heads) * head_dim;
    const Span QKV = span(qkv, static_cast<size_t>(n_tokens * width) * 2);
    const Span ins[4] = {span(positions, static_cast<size_t>(n_tokens) * 8),
                         span(cos_sin_cache, static_cast<size_t>(max_positions * head_dim) * 4),
                         span(q_weight, static_cast<size_t>(head_dim) * 2), span(k_weight, static_cast<size_t>(head_dim) * 2)};
    for (const Span& i : ins)
        if (overlaps(QKV, i)) return RMSQ_ERR_ALIAS;
    const int st = check_device();
    if (st != RMSQ_OK) return st;
    rmsq::QkLaunch l;
    l.qkv = qkv;
    l.positions = positions;
    l.cos_sin = cos_sin_cache;
    l.max_pos = max_positions;
    l.q_weight = q_weight;
    l.k_weight = k_weight;
    l.eps = eps;
    l.n = static_cast<int>(n_tokens);
    l.nq = num_q_heads;
    l.nkv = num_kv_heads;
    l.head_dim = head_dim;
    l.neox = is_neox == 1;
    l.fp16 = dtype == RMSQ_FP16;
    l.variant = variant == RMSQ_VARIANT_DIRECT ? rmsq::kVariantDirect
                : variant == RMSQ_VARIANT_PIPELINED ? rmsq::kVariantPipelined : rmsq::kVariantAuto;
    const cudaError_t e = rmsq::launch_qk_norm_rope(l, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RMSQ_OK : fail_cuda(e);
}

int rmsq_qk_norm_rope(void* qkv, const int64_t* positions, const float* cos_sin_cache, int64_t max_positions,
                      const void* q_weight, const void* k_weight, float eps, int64_t n_tokens, int num_q_heads,
                      int num_kv_heads, int head_dim, int is_neox, int dtype, void* stream) {
    return rmsq_qk_norm_rope_ex(qkv, positions, cos_sin_cache, max_positions, q_weight, k_weight, eps, n_tokens,
                                num_q_heads, num_kv_heads, head_dim, is_neox, dtype, stream, RMSQ_VARIANT_AUTO);
}

size_t rmsq_nvfp4_dynamic_workspace_bytes(int64_t n_tokens) {
    return n_tokens < 0 ? 0 : rmsq::nvfp4_dynamic_workspace_bytes(n_tokens);
}

int rmsq_fused_add_rmsnorm_nvfp4_dynamic(const void* x, const void* residual, const void* weight,
                                         float eps, void* out_q, void* out_block_scales,
                                         float* out_global_scale, void* residual_out, void* workspace,
                                         size_t workspace_bytes, int64_t n_tokens, int64_t hidden,
                                         int dtype, void* stream, int variant) {
    if (dtype != RMSQ_BF16 && dtype != RMSQ_FP16) return RMSQ_ERR_INVALID_ARG;
    if (variant != RMSQ_VARIANT_AUTO && variant != RMSQ_VARIANT_DIRECT && variant != RMSQ_VARIANT_PIPELINED)
        return RMSQ_ERR_INVALID_ARG;
    int st = check_shape(RMSQ_NVFP4, n_tokens, hidden);
    if (st != RMSQ_OK) return st;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSQ_ERR_INVALID_ARG;
    if (n_tokens == 0) return RMSQ_OK;
    if (!x || !weight || !out_q || !out_block_scales || !out_global_scale || !workspace)
        return RMSQ_ERR_INVALID_ARG;
    if ((residual == nullptr) != (residual_out == nullptr)) return RMSQ_ERR_INVALID_ARG;
    const size_t ws_need = rmsq::nvfp4_dynamic_workspace_bytes(n_tokens);
    if (workspace_bytes < ws_need) return RMSQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(weight, 16) || !aligned(residual_out, 16) ||
        !aligned(out_q, 16) || !aligned(out_global_scale, 4) || !aligned(workspace, 16))
        return RMSQ_ERR_ALIGNMENT;
    size_t q_bytes = 0, sc_bytes = 0;
    sizes_of(RMSQ_NVFP4, n_tokens, hidden, &q_bytes, &sc_bytes);
    const size_t act = static_cast<size_t>(n_tokens * hidden) * 2;
    const Span X = span(x, act), R = span(residual, act), W = span(weight, hidden * 2),
               RO = span(residual_out, act), Q = span(out_q, q_bytes), SC = span(out_block_scales, sc_bytes),
               GS = span(out_global_scale, 4), WS = span(workspace, ws_need);
    if (residual && X.lo != R.lo && overlaps(X, R)) return RMSQ_ERR_ALIAS;
    if (residual_out) {
        if (RO.lo != X.lo && overlaps(RO, X)) return RMSQ_ERR_ALIAS;
        if (RO.lo != R.lo && overlaps(RO, R)) return RMSQ_ERR_ALIAS;
        if (overlaps(RO, W)) return RMSQ_ERR_ALIAS;
    }
    const Span outs[4] = {Q, SC, GS, WS};
    for (int i = 0; i < 4; ++i) {
        const Span& o = outs[i];
        if (overlaps(o, X) || overlaps(o, R) || overlaps(o, W) || overlaps(o, RO)) return RMSQ_ERR_ALIAS;
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(o, outs[j])) return RMSQ_ERR_ALIAS;
    }
    st = check_device();
    if (st != RMSQ_OK) return st;

    rmsq::LaunchArgs la = {};
    la.x = x;
    la.res = residual;
    la.w = weight;
    la.res_out = residual_out;
    la.q = out_q;
    la.scales = out_block_scales;
    la.scale_in = nullptr;
    la.eps = eps;
    la.mode = RMSQ_NVFP4;
    la.n = static_cast<int>(n_tokens);
    la.hidden = static_cast<int>(hidden);
    la.variant = variant == RMSQ_VARIANT_DIRECT ? rmsq::kVariantDirect
                 : variant == RMSQ_VARIANT_PIPELINED ? rmsq::kVariantPipelined : rmsq::kVariantAuto;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == RMSQ_BF16
                              ? rmsq::launch_nvfp4_dynamic_bf16(la, workspace, out_global_scale, s)
                              : rmsq::launch_nvfp4_dynamic_fp16(la, workspace, out_global_scale, s);
    return e == cudaSuccess ? RMSQ_OK : fail_cuda(e);
}

int rmsq_fused_add_rmsnorm_quant(const void* x, const void* residual, const void* weight, float eps,
                                 int quant_mode, const float* scale_in, void* out_q, void* out_scales,
                                 void* residual_out, int64_t n_tokens, int64_t hidden, int dtype,
                                 void* stream) {
    return rmsq_fused_add_rmsnorm_quant_ex(x, residual, weight, eps, quant_mode, scale_in, out_q,
                                           out_scales, residual_out, n_tokens, hidden, dtype, stream,
                                           RMSQ_VARIANT_AUTO);
}

int rmsq_take_fault_flags(uint32_t* flags) {
    if (!flags) return RMSQ_ERR_INVALID_ARG;
    const int st = check_device();
    if (st != RMSQ_OK) return st;
    unsigned int a = 0, b = 0, c = 0, d = 0;
    cudaError_t e = rmsq::take_pipe_fault_bf16(&a);
    if (e == cudaSuccess) e = rmsq::take_pipe_fault_fp16(&b);
    if (e == cudaSuccess) e = rmsq::take_pipe_fault_qk(&c);
    if (e == cudaSuccess) e = rmsq::take_pipe_fault_ar(&d);
    if (e != cudaSuccess) return fail_cuda(e);
    *flags = a | b | c | d;
    return RMSQ_OK;
}

int rmsq_query_sizes(int quant_mode, int64_t n_tokens, int64_t hidden, size_t* q_bytes,
                     size_t* scale_bytes) {
    if (!q_bytes || !scale_bytes) return RMSQ_ERR_INVALID_ARG;
    const int st = check_shape(quant_mode, n_tokens, hidden);
    if (st != RMSQ_OK) return st;
    sizes_of(quant_mode, n_tokens, hidden, q_bytes, scale_bytes);
    return RMSQ_OK;
}

int rmsq_debug_convert(int kind, const float* in, uint8_t* out, int64_t n, void* stream) {
    if ((kind != 0 && kind != 1) || n < 0) return RMSQ_ERR_INVALID_ARG;
    if (n == 0) return RMSQ_OK;
    if (!in || !out) return RMSQ_ERR_INVALID_ARG;
    if (!aligned(in, 4)) return RMSQ_ERR_ALIGNMENT;
    if (overlaps(span(in, static_cast<size_t>(n) * 4), span(out, static_cast<size_t>(n))))
        return RMSQ_ERR_ALIAS;
    const int st = check_device();
    if (st != RMSQ_OK) return st;
    const cudaError_t e = rmsq::launch_convert(kind, in, out, n, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RMSQ_OK : fail_cuda(e);
}

int rmsq_debug_activation(int kind, const float* in, const float* in2, float* out, int64_t n, void* stream) {
    if (kind < 0 || kind > 3 || n < 0) return RMSQ_ERR_INVALID_ARG;
    if (n == 0) return RMSQ_OK;
    if (!in || !out || (kind == 2 && !in2)) return RMSQ_ERR_INVALID_ARG;
    if (kind != 2) in2 = nullptr;
    if (!aligned(in, 4) || !aligned(in2, 4) || !aligned(out, 4)) return RMSQ_ERR_ALIGNMENT;
    const Span O = span(out, static_cast<size_t>(n) * 4);
    if (overlaps(O, span(in, static_cast<size_t>(n) * 4)) || overlaps(O, span(in2, static_cast<size_t>(n) * 4)))
        return RMSQ_ERR_ALIAS;
    const int st = check_device();
    if (st != RMSQ_OK) return st;
    const cudaError_t e = rmsq::launch_debug_activation(kind, in, in2, out, n, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RMSQ_OK : fail_cuda(e);
}

int rmsq_debug_bounded_wait(int64_t limit_ns, int* gave_up) {
    if (limit_ns <= 0 || limit_ns > 1000000000 || !gave_up) return RMSQ_ERR_INVALID_ARG;
    const int st = check_device();
    if (st != RMSQ_OK) return st;
    const cudaError_t e = rmsq::debug_bounded_wait(static_cast<uint64_t>(limit_ns), gave_up);
    return e == cudaSuccess ? RMSQ_OK : fail_cuda(e);
}

const char* rmsq_status_string(int status) {
    switch (status) {
    case RMSQ_OK: return "ok";
    case RMSQ_ERR_INVALID_ARG: return "invalid argument";
    case RMSQ_ERR_ALIGNMENT: return "misaligned pointer";
    case RMSQ_ERR_ALIAS: return "overlapping buffers";
    case RMSQ_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case RMSQ_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case RMSQ_ERR_NO_DEVICE: return "no CUDA device";
    case RMSQ_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
    }
}

int rmsq_last_cuda_error(void) { return t_last_cuda_error; }

int rmsq_version(void) { return RMSQ_VERSION; }

}  // extern "C"

// Picks and launches a row-kernel instantiation for (mode, residual, chunks
// per thread J, variant).  Included once per activation type.
//
//  direct:    one CTA per row, ceil(hidden / 8 / J) threads (J = 1 up to
//             hidden 8192, else 2; also 2 when the rows would not all be
//             resident at once with J = 1), loads straight into registers.
//  pipelined: persistent CTAs (as many as fit on the SMs), `stages` rows of
//             x / residual in flight per CTA through the shared-memory ring.
//             The per-row dependency chain (block reductions, IEEE divide
//             and square root) rather than bytes in flight limits a CTA, so
//             more CTAs per SM beat a deeper ring (measured on GB300): two
//             stages and J = 2 with a residual (4 without) when the CTAs get
//             few rows each, one stage and J = 4 (8 without a residual) from
//             8 rows per CTA on (plan_rows); J doubled while a row would need
//             more than 512 threads.
#pragma once

#include <atomic>
#include <mutex>

#include "rmsq_launch.h"
#include "rmsq_nvfp4_dyn.cuh"
#include "rmsq_pipe.cuh"
#include "rmsq_rows.cuh"

namespace rmsq {

static_assert(kModeNormOnly == kNormOnly, "host and kernel codes of the norm-only mode");

// Set by a pipelined CTA that gave up waiting for its copies (this unit's
// instantiations only).
static __device__ unsigned int g_pipe_fault;

// Compile-time tuning (results never depend on these): the minimum number of
// resident 512-thread CTAs the pipelined kernel is compiled for when a thread
// owns one or two chunks, with and without a residual (the register budget
// follows from it: 1 leaves up to 128 registers, 2 caps them at 64), and
// whether the largest shared-memory carve-out is requested.  Without a
// residual the kernel is bound by its instruction stream rather than by HBM,
// and the extra resident CTAs of the tighter budget pay (measured on GB300);
// with a residual they do not.
#ifndef RMSQ_PIPE_MIN_BLOCKS
#define RMSQ_PIPE_MIN_BLOCKS 1
#endif
#ifndef RMSQ_PIPE_MIN_BLOCKS_NORES
#define RMSQ_PIPE_MIN_BLOCKS_NORES 2
#endif
#ifndef RMSQ_MAX_SMEM_CARVEOUT
#define RMSQ_MAX_SMEM_CARVEOUT 1
#endif
// Paired (32-byte) activation accesses where the buffers allow them.
#ifndef RMSQ_PAIR_ACCESS
#define RMSQ_PAIR_ACCESS 1
#endif

// Register budget of the pipelined kernel by chunks per thread (compile-time
// tuning, results do not depend on it): with four chunks per thread the
// natural allocation (~86) leaves five 128-thread CTAs per SM; 80 gives six.
// NVFP4 with two chunks per thread: a cap of 64 (the allocation drops from
// 68 to 56) lets nine 128-thread CTAs share an SM instead of seven
// (Qwen3-shaped layer, hidden 2048, 16384 rows: 36.1 -> 35.3 us); the FP8
// modes at two chunks per thread were 3-5 % slower under that cap (hidden
// 4096), so they keep the natural allocation.
#ifndef RMSQ_PIPE_MAXNREG_J4
#define RMSQ_PIPE_MAXNREG_J4 80
#endif
#ifndef RMSQ_PIPE_MAXNREG_J8
#define RMSQ_PIPE_MAXNREG_J8 128
#endif
#ifndef RMSQ_PIPE_MAXNREG_NVFP4_J2
#define RMSQ_PIPE_MAXNREG_NVFP4_J2 64
#endif
template <int J> constexpr int pipe_maxnreg() {
    return J == 4 ? RMSQ_PIPE_MAXNREG_J4 : J == 8 ? RMSQ_PIPE_MAXNREG_J8 : 128;
}
template <int MODE, int J> constexpr int pipe_mode_maxnreg() {
    return (MODE == kNvfp4 && J == 2) ? RMSQ_PIPE_MAXNREG_NVFP4_J2 : pipe_maxnreg<J>();
}

template <class E, int MODE, bool RES, int J>
__global__ void __launch_bounds__(kPipeMaxThreads) __maxnreg__((pipe_mode_maxnreg<MODE, J>()))
pipe_entry(const RowArgs a, const int stages) {
    pipe_body<E, MODE, RES, J>(a, stages, &g_pipe_fault);
}

template <class E, int MODE, bool RES>
const void* pick_direct(int J) {
    if (J == 1) return reinterpret_cast<const void*>(&rows_kernel<E, MODE, RES, 1>);
    return reinterpret_cast<const void*>(&rows_kernel<E, MODE, RES, 2>);
}

template <class E, int MODE, bool RES>
const void* pick_pipe(int J) {
    switch (J) {
    case 1: return reinterpret_cast<const void*>(&pipe_entry<E, MODE, RES, 1>);
    case 2: return reinterpret_cast<const void*>(&pipe_entry<E, MODE, RES, 2>);
    case 4: return reinterpret_cast<const void*>(&pipe_entry<E, MODE, RES, 4>);
    default: return reinterpret_cast<const void*>(&pipe_entry<E, MODE, RES, 8>);
    }
}

template <class E, int MODE>
const void* pick_res(bool res, bool pipe, int J) {
    if (pipe) return res ? pick_pipe<E, MODE, true>(J) : pick_pipe<E, MODE, false>(J);
    return res ? pick_direct<E, MODE, true>(J) : pick_direct<E, MODE, false>(J);
}

template <class E>
const void* pick_kernel(int mode, bool res, bool pipe, int J) {
    switch (mode) {
    case kFp8Static: return pick_res<E, kFp8Static>(res, pipe, J);
    case kFp8PerToken: return pick_res<E, kFp8PerToken>(res, pipe, J);
    case kFp8G128Row: return pick_res<E, kFp8G128Row>(res, pipe, J);
    case kFp8G128Col: return pick_res<E, kFp8G128Col>(res, pipe, J);
    case kFp8G64Row: return pick_res<E, kFp8G64Row>(res, pipe, J);
    case kFp8G64Col: return pick_res<E, kFp8G64Col>(res, pipe, J);
    case kNvfp4: return pick_res<E, kNvfp4>(res, pipe, J);
    case kNormAmax: return pick_res<E, kNormAmax>(res, pipe, J);
    case kNormOnly: return pick_res<E, kNormOnly>(res, pipe, J);
    default: return nullptr;
    }
}

// One kernel launch, with programmatic stream serialisation unless it is
// switched off: the kernel may then start while the previous kernel of the
// stream finishes; the kernels wait for it before any memory access.
inline cudaError_t launch_kernel(const void* fn, dim3 grid, dim3 block, void** params, size_t smem,
                                 cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic_launch() ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, params);
}

// Occupancy of a pipelined instantiation for a given ring size, cached per
// device.
struct OccEntry {
    int dev;
    const void* fn;
    int smem;
    int threads;
    int blocks;
};

// Shared-memory ring budget per CTA (two CTAs per SM).
constexpr int kPipeSmemBudget = 110 * 1024;

// The largest dynamic shared memory a CTA of `fn` may use on the current
// device: the per-block opt-in maximum less the function's static shared
// memory (cached per device and function; neither changes with a context
// reset).
inline int dyn_smem_limit(const void* fn, cudaError_t* err) {
    struct Entry {
        int dev;
        const void* fn;
        int limit;
    };
    static std::mutex mu;
    static Entry cache[256];
    static int used = 0;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].fn == fn) return cache[i].limit;
    int optin = 0;
    *err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (*err != cudaSuccess) return 0;
    cudaFuncAttributes fa;
    *err = cudaFuncGetAttributes(&fa, fn);
    if (*err != cudaSuccess) return 0;
    const int limit = optin - static_cast<int>(fa.sharedSizeBytes);
    if (used < 256) cache[used++] = {dev, fn, limit};
    return limit;
}

// The opt-in dynamic shared memory limit of a pipelined instantiation (the
// largest a CTA may use, so that no launch ever lowers it below what another
// launch of the same function needs) and its carve-out preference.  Function
// attributes belong to the context of the current device, so they are set
// before every launch (a host-side call, no device work): a second device, or
// a device whose primary context was reset, never gets a launch without them.
inline cudaError_t set_smem_attributes(const void* fn) {
    cudaError_t e = cudaSuccess;
    const int limit = dyn_smem_limit(fn, &e);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    // Prefer the largest shared-memory carve-out so that the rings of several
    // CTAs fit on one SM (the kernels barely use L1: loads bypass it).
    if (e == cudaSuccess && RMSQ_MAX_SMEM_CARVEOUT)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

// Resident CTAs per SM of `fn` at `threads` threads and `smem` dynamic
// shared-memory bytes (cached per device and launch shape).
inline int occupancy_blocks(const void* fn, int threads, int smem, cudaError_t* err) {
    static std::mutex mu;
    constexpr int kCache = 256;   // more than the launch shapes in use; beyond it, queried per call
    static OccEntry cache[kCache];
    static int used = 0;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].fn == fn && cache[i].smem == smem && cache[i].threads == threads)
            return cache[i].blocks;
    int blocks = 0;
    *err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, threads, smem);
    if (*err != cudaSuccess) return 0;
    if (used < kCache) cache[used++] = {dev, fn, smem, threads, blocks};
    return blocks;
}

// The same for a pipelined kernel, whose shared-memory attributes are set
// first.
inline int pipe_blocks_per_sm(const void* fn, int threads, int smem, cudaError_t* err) {
    *err = set_smem_attributes(fn);
    if (*err != cudaSuccess) return 0;
    return occupancy_blocks(fn, threads, smem, err);
}

inline int sm_count(cudaError_t* err) {
    static std::atomic<int> cached[128];
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess || dev < 0 || dev >= 128) return 0;
    int v = cached[dev].load(std::memory_order_acquire);
    if (v == 0) {
        *err = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (*err != cudaSuccess) return 0;
        cached[dev].store(v, std::memory_order_release);
    }
    return v;
}

// Default ring: two stages (one row computed while the next is in flight),
// one when two do not fit the budget.
inline int pipe_stages(int stage_bytes) { return 2 * stage_bytes <= kPipeSmemBudget ? 2 : 1; }

inline RowArgs make_row_args(const LaunchArgs& la) {
    RowArgs a;
    a.x = static_cast<const uint4*>(la.x);
    a.res = static_cast<const uint4*>(la.res);
    a.w = static_cast<const uint4*>(la.w);
    a.res_out = static_cast<uint4*>(la.res_out);
    a.q = static_cast<uint8_t*>(la.q);
    a.scales = la.scales;
    a.scale_in = la.scale_in;
    a.eps = la.eps;
    a.n = la.n;
    a.hidden = la.hidden;
    a.chunks = la.hidden / 8;
    a.inv_hidden_pow2 = (la.hidden & (la.hidden - 1)) == 0 ? 1.0f / (float)la.hidden : 0.0f;
    auto on = [](const void* p, uintptr_t b) { return p == nullptr || reinterpret_cast<uintptr_t>(p) % b == 0; };
    a.pair = RMSQ_PAIR_ACCESS && a.chunks % 2 == 0 && on(la.x, 32) && on(la.res, 32) &&
             on(la.res_out, 32) && on(la.q, 16);
    a.e8m0 = la.e8m0;
    a.ue8m0 = la.ue8m0;
    a.col_stride = la.col_stride;
    return a;
}

// Launch shape of the pipelined kernel: chunks per thread J, threads, ring
// stages and bytes.
struct PipePlan {
    int J, threads, stages, smem;
};

// Chunks per thread by default (measured on GB300): with a residual the
// kernel is bound by HBM and two chunks per thread (more threads per row,
// more loads in flight) are fastest; without one it is bound by instruction
// issue, and four chunks per thread from 256 chunks (hidden 2048) up spread a
// warp's fixed per-row work (reductions, inverse RMS, scale) over 1024
// elements.
inline int pipe_default_j(int chunks, bool res) { return (!res && chunks >= 256) ? 4 : 2; }

// Chunks per thread when the CTAs have many rows each (below): four with a
// residual above hidden 2048, eight without from hidden 4096 (else as the
// default).
inline int pipe_many_rows_j(int chunks, bool res) {
    if (res) return chunks > 256 ? 4 : 2;
    return chunks >= 512 ? 8 : pipe_default_j(chunks, res);
}

// The plan for J chunks per thread (doubled while a row would need more than
// 512 threads) and `stages` ring stages (fewer if the ring would not fit the
// budget).
inline PipePlan make_pipe_plan(const RowArgs& a, bool res, int J, int stages) {
    auto threads_for = [&](int j) { return ((a.chunks + 32 * j - 1) / (32 * j)) * 32; };
    PipePlan p;
    p.J = J;
    while (p.J < 8 && threads_for(p.J) > kPipeMaxThreads) p.J *= 2;
    p.threads = threads_for(p.J);
    const int stage_bytes = a.chunks * 16 * (res ? 2 : 1);   // x (+ residual) of one row
    p.stages = stages;
    while (p.stages > 1 && p.stages * stage_bytes > kPipeSmemBudget) --p.stages;
    // The weights (four or eight chunks per thread) sit after the ring.
    p.smem = p.stages * stage_bytes + co_weight_smem_bytes(p.J, p.threads * p.J);
    return p;
}

inline PipePlan pipe_plan(const RowArgs& a, bool res) {
    const PipeTuning tune = get_pipe_tuning();
    auto threads_for = [&](int j) { return ((a.chunks + 32 * j - 1) / (32 * j)) * 32; };
    int J = pipe_default_j(a.chunks, res);
    const int tj = tune.chunks_per_thread;
    if ((tj == 1 || tj == 2 || tj == 4 || tj == 8) && threads_for(tj) <= kPipeMaxThreads) J = tj;
    const int stage_bytes = a.chunks * 16 * (res ? 2 : 1);
    int stages = pipe_stages(stage_bytes);
    if (tune.stages >= 1 && tune.stages <= kMaxStages && tune.stages * stage_bytes <= kPipeSmemBudget)
        stages = tune.stages;
    return make_pipe_plan(a, res, J, stages);
}

// Persistent grid of `fn` for a plan: as many CTAs as fit on the SMs at once
// (capped by the tuning), at most one per row.
inline cudaError_t pipe_grid(const void* fn, const PipePlan& p, int n, int* grid) {
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (err != cudaSuccess) return err;
    int per_sm = pipe_blocks_per_sm(fn, p.threads, p.smem, &err);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const PipeTuning tune = get_pipe_tuning();
    if (tune.ctas_per_sm >= 1 && tune.ctas_per_sm < per_sm) per_sm = tune.ctas_per_sm;
    *grid = n < per_sm * sms ? n : per_sm * sms;
    return cudaSuccess;
}

// Rows per CTA from which the many-rows plan is taken.
constexpr int kManyRowsPerCta = 8;

// The launch of the row work for `la`: kernel, grid, block, plan.
struct RowLaunch {
    bool pipe;
    const void* fn;
    int grid, threads, smem, stages, J;
};

// Chooses the variant (direct kernel below kPipeMinRowsPerSm rows per SM,
// unless one is forced) and, for the pipelined kernel, the plan (measured on
// GB300): when each CTA of the persistent grid gets at least
// kManyRowsPerCta rows, a one-stage ring with pipe_many_rows_j chunks per
// thread, whose smaller CTAs and rings let more CTAs share an SM (hidden
// 7168 with a residual, 8192 rows: 71.4 -> 68.9 us; hidden 8192: 53 -> 40
// us; Qwen-shaped NVFP4, 16384 rows: 37.3 -> 36.0 us); with fewer rows per
// CTA the two-stage ring's head start at the kernel's beginning weighs more
// and pipe_plan's default stays (Llama- and Qwen-shaped layers of 4096
// rows).  A tuning setting of the chunks per thread or the stages keeps
// pipe_plan as tuned.
template <class E>
cudaError_t plan_rows(const LaunchArgs& la, const RowArgs& a, RowLaunch* out) {
    const bool res = la.res != nullptr;
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (err != cudaSuccess) return err;
    out->pipe = la.variant == kVariantPipelined ||
                (la.variant == kVariantAuto && a.n >= kPipeMinRowsPerSm * sms);
    if (!out->pipe) {
        auto threads_for = [&](int j) { return ((a.chunks + j - 1) / j + 31) / 32 * 32; };
        out->J = a.chunks <= 1024 ? 1 : 2;
        out->fn = pick_kernel<E>(la.mode, res, false, out->J);
        if (!out->fn) return cudaErrorInvalidValue;
        if (out->J == 1 && a.chunks >= 2 && a.n > sms) {
            // One CTA per row (measured on GB300, 256 rows of hidden 8192):
            // when the rows do not all fit on the SMs at once with one chunk
            // per thread, two chunks per thread (half the threads, so more
            // CTAs per SM) finish in fewer waves; without a residual they
            // are also faster once SMs hold two rows (static and group
            // scales 7-10 %; with a residual the same or 2 % slower).
            const int per_sm1 = occupancy_blocks(out->fn, threads_for(1), 0, &err);
            if (err != cudaSuccess) return err;
            const void* f2 = pick_kernel<E>(la.mode, res, false, 2);
            if (!f2) return cudaErrorInvalidValue;
            const int per_sm2 = occupancy_blocks(f2, threads_for(2), 0, &err);
            if (err != cudaSuccess) return err;
            const bool waves = (int64_t)a.n > (int64_t)per_sm1 * sms && per_sm2 > per_sm1;
            if (waves || (!res && per_sm2 >= per_sm1)) {
                out->J = 2;
                out->fn = f2;
            }
        }
        out->threads = threads_for(out->J);
        out->grid = a.n;
        out->smem = 0;
        out->stages = 0;
        return cudaSuccess;
    }
    const PipeTuning tune = get_pipe_tuning();
    PipePlan p = pipe_plan(a, res);
    const void* fn = pick_kernel<E>(la.mode, res, true, p.J);
    if (!fn) return cudaErrorInvalidValue;
    int grid = 0;
    err = pipe_grid(fn, p, a.n, &grid);
    if (err != cudaSuccess) return err;
    if (tune.chunks_per_thread == 0 && tune.stages == 0) {
        const PipePlan q = make_pipe_plan(a, res, pipe_many_rows_j(a.chunks, res), 1);
        const void* fq = pick_kernel<E>(la.mode, res, true, q.J);
        int gq = 0;
        if (!fq) return cudaErrorInvalidValue;
        err = pipe_grid(fq, q, a.n, &gq);
        if (err != cudaSuccess) return err;
        if ((int64_t)a.n >= (int64_t)kManyRowsPerCta * gq) {
            p = q;
            fn = fq;
            grid = gq;
        }
    }
    out->fn = fn;
    out->grid = grid;
    out->threads = p.threads;
    out->smem = p.smem;
    out->stages = p.stages;
    out->J = p.J;
    return cudaSuccess;
}

// One launch of the row work; *grid_out (if given) receives the number of
// CTAs launched.
template <class E>
cudaError_t launch_rows(const LaunchArgs& la, cudaStream_t stream, int* grid_out = nullptr) {
    RowArgs a = make_row_args(la);
    RowLaunch l;
    const cudaError_t err = plan_rows<E>(la, a, &l);
    if (err != cudaSuccess) return err;
    if (grid_out) *grid_out = l.grid;
    if (l.pipe) {
        int st = l.stages;
        void* params[] = {&a, &st};
        return launch_kernel(l.fn, dim3(l.grid), dim3(l.threads), params, l.smem, stream);
    }
    void* params[] = {&a};
    return launch_kernel(l.fn, dim3(l.grid), dim3(l.threads), params, 0, stream);
}

// The launch launch_rows would make for `la` (no launch).
template <class E>
cudaError_t query_rows(const LaunchArgs& la, RowLaunch* out) {
    const RowArgs a = make_row_args(la);
    return plan_rows<E>(la, a, out);
}

// NVFP4 with a data-derived global scale: pass 1 (row kernel, mode
// kNormAmax, in the requested variant), pass 2 (block quantisation), both
// launched with programmatic dependent launch when it is on, so pass 2
// overlaps the end of pass 1 and waits for it before touching memory.
template <class E>
cudaError_t launch_nvfp4_dynamic(const LaunchArgs& la, void* workspace, float* out_gs,
                                 cudaStream_t stream) {
    LaunchArgs first = la;
    first.mode = kNormAmax;
    first.q = nullptr;
    first.scales = workspace;
    first.scale_in = nullptr;
    int parts = 0;
    cudaError_t e = launch_rows<E>(first, stream, &parts);
    if (e != cudaSuccess) return e;
    const int sms = sm_count(&e);
    if (e != cudaSuccess) return e;
    const void* fn = reinterpret_cast<const void*>(&nvfp4_dyn_quant_kernel<E>);
    int per_sm = kDynCtasPerSm;
    if (per_sm <= 0) per_sm = occupancy_blocks(fn, 256, 0, &e);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int rows_per_sweep = 0, threads = 0;
    nvfp4_dyn_shape(la.n, la.hidden, (int64_t)sms * per_sm * 256, &rows_per_sweep, &threads);
    const int64_t grid = ((int64_t)threads + 255) / 256;
    auto at32 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 32 == 0; };
    const uint4* h = static_cast<const uint4*>(la.res ? la.res_out : la.x);
    const uint4* w = static_cast<const uint4*>(la.w);
    int pair = (RMSQ_PAIR_ACCESS && at32(h)) ? 1 : 0;
    const float* ws = static_cast<const float*>(workspace);
    uint2* q = static_cast<uint2*>(la.q);
    uint8_t* bs = static_cast<uint8_t*>(la.scales);
    int n = la.n, hidden = la.hidden;
    void* params[] = {&h, &w, &ws, &q, &bs, &out_gs, &n, &hidden, &pair, &parts, &rows_per_sweep, &threads};
    return launch_kernel(fn, dim3((unsigned)grid), dim3(256), params, 0, stream);
}

// Reads and clears this unit's pipeline fault flag (current device).
inline cudaError_t take_pipe_fault(unsigned int* out) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_pipe_fault, sizeof(unsigned int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_pipe_fault, &zero, sizeof(unsigned int));
    return e;
}

}  // namespace rmsq

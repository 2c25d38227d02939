// All-reduce + residual add + RMSNorm + quantisation in one kernel (vLLM docs
// "Fusion torch.compile passes", section "AllReduce + RMSNorm
// (fuse_allreduce_rms)": the tensor-parallel all-reduce fused with the
// following residual add, RMSNorm and optional FP8 / NVFP4 quantisation, used
// at small token counts).
//
// The all-reduce is done one-shot, by loads: every row's partial sums are read
// from each rank's buffer (peer memory over NVLink on a multi-GPU node, or
// any buffers the current device can address), added in rank order in fp32
// and rounded once to the activation type; that row is the x of the fused op,
// and the rest of the row is the row kernels' arithmetic (rmsq_rowmath.cuh),
// bit for bit.  Two kernels: one CTA per row, every load issued up front into
// registers (ar_rows_kernel), and the pipelined kernel (pipe_body with AR:
// persistent CTAs, each ring stage holding the ranks' partial rows and the
// residual row, copied in by bulk asynchronous copies) from kPipeMinRowsPerSm
// rows per SM with up to kArPipeMaxRanks ranks.  No kernel waits on another GPU: the caller
// orders the launch after every rank's partials are complete.
#include "rmsq_dispatch.cuh"

namespace rmsq {

// x = T(sum over ranks of fp32(partial)) for the thread's chunks, in rank
// order, one rounding at the end.
template <class E, int J>
__device__ __forceinline__ void ar_load_sum(const ArRanks& rk, int64_t base, int c0, int chunks, uint4 (&xv)[J]) {
    uint4 pv[kMaxArRanks][J];
#pragma unroll
    for (int r = 0; r < kMaxArRanks; ++r)
#pragma unroll
        for (int j = 0; j < J; ++j) {
            pv[r][j] = make_uint4(0u, 0u, 0u, 0u);
            if (r < rk.n && c0 + j < chunks) pv[r][j] = ld_act(rk.part[r] + base + c0 + j);
        }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        float acc[8];
        const uint32_t w0[4] = {pv[0][j].x, pv[0][j].y, pv[0][j].z, pv[0][j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) { acc[2 * k] = E::lo(w0[k]); acc[2 * k + 1] = E::hi(w0[k]); }
#pragma unroll
        for (int r = 1; r < kMaxArRanks; ++r) {
            if (r >= rk.n) break;
            const uint32_t wr[4] = {pv[r][j].x, pv[r][j].y, pv[r][j].z, pv[r][j].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 s = add2_rn(make_float2(acc[2 * k], acc[2 * k + 1]), make_float2(E::lo(wr[k]), E::hi(wr[k])));
                acc[2 * k] = s.x;
                acc[2 * k + 1] = s.y;
            }
        }
        xv[j] = make_uint4(E::pack(acc[0], acc[1]), E::pack(acc[2], acc[3]), E::pack(acc[4], acc[5]),
                           E::pack(acc[6], acc[7]));
    }
}

template <class E, int MODE, bool RES, int J>
__global__ void __launch_bounds__(1024) ar_rows_kernel(const RowArgs a, const ArRanks rk) {
    __shared__ __align__(16) float s_sum[32];
    __shared__ float s_max[32];
    if (threadIdx.x < 32 && (int)threadIdx.x >= (int)(blockDim.x >> 5)) s_sum[threadIdx.x] = 0.0f;
    allow_dependents();
    grid_dependency_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int row = blockIdx.x;
    const int64_t base = (int64_t)row * a.chunks;
    const int c0 = tid * J;

    uint4 xv[J], rv[J], wv[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        rv[j] = wv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (c0 + j < a.chunks) {
            wv[j] = ld_weight(a.w + c0 + j);
            if constexpr (RES) rv[j] = ld_act(a.res + base + c0 + j);
        }
    }
    ar_load_sum<E, J>(rk, base, c0, a.chunks, xv);
    const float sin = ModeTraits<MODE>::needs_scale_in ? __ldg(a.scale_in) : 0.0f;
    __shared__ float s_rtab[MODE == kNvfp4 ? 128 : 1];
    if constexpr (MODE == kNvfp4) fill_nvfp4_rtab(s_rtab, sin);   // ordered by the barrier below

    uint32_t h[J][4];
    float acc = combine_chunks<E, RES, J>(xv, rv, h, a.res_out + base, c0, a.chunks, false);
    acc = warp_tree_sum(acc);
    if (lane == 0) s_sum[warp] = acc;
    __syncthreads();
    const float inv = inv_rms(warp_slots_tree_sum<32>(s_sum, nwarps), a);
    float run_max = 0.0f;
    float wf[J][8];
    widen_weights<E, J>(wv, wf);
    quantize_row<E, MODE, J>(a, row, h, wf, inv, sin, s_rtab, s_max, tid, nwarps, run_max);
}

template <class E, int MODE, bool RES>
const void* pick_ar(int J) {
    return J == 1 ? reinterpret_cast<const void*>(&ar_rows_kernel<E, MODE, RES, 1>)
                  : reinterpret_cast<const void*>(&ar_rows_kernel<E, MODE, RES, 2>);
}

template <class E, int MODE>
const void* pick_ar_res(bool res, int J) {
    return res ? pick_ar<E, MODE, true>(J) : pick_ar<E, MODE, false>(J);
}

template <class E>
const void* pick_ar_kernel(int mode, bool res, int J) {
    switch (mode) {
    case kFp8Static: return pick_ar_res<E, kFp8Static>(res, J);
    case kFp8PerToken: return pick_ar_res<E, kFp8PerToken>(res, J);
    case kFp8G128Row: return pick_ar_res<E, kFp8G128Row>(res, J);
    case kFp8G128Col: return pick_ar_res<E, kFp8G128Col>(res, J);
    case kFp8G64Row: return pick_ar_res<E, kFp8G64Row>(res, J);
    case kFp8G64Col: return pick_ar_res<E, kFp8G64Col>(res, J);
    case kNvfp4: return pick_ar_res<E, kNvfp4>(res, J);
    default: return nullptr;
    }
}

// The pipelined all-reduce kernel.
template <class E, int MODE, bool RES, int J>
__global__ void __launch_bounds__(kPipeMaxThreads) __maxnreg__(pipe_maxnreg<J>())
pipe_ar_entry(const RowArgs a, const int stages, const __grid_constant__ ArRanks rk) {
    pipe_body<E, MODE, RES, J, true>(a, stages, &g_pipe_fault, &rk);
}

template <class E, int MODE, bool RES>
const void* pick_ar_pipe_j(int J) {
    return J == 2 ? reinterpret_cast<const void*>(&pipe_ar_entry<E, MODE, RES, 2>)
                  : reinterpret_cast<const void*>(&pipe_ar_entry<E, MODE, RES, 4>);
}

template <class E>
const void* pick_ar_pipe(int mode, bool res, int J) {
    switch (mode) {
#define RMSQ_AR_PIPE_CASE(M) \
    case M: return res ? pick_ar_pipe_j<E, M, true>(J) : pick_ar_pipe_j<E, M, false>(J);
    RMSQ_AR_PIPE_CASE(kFp8Static)
    RMSQ_AR_PIPE_CASE(kFp8PerToken)
    RMSQ_AR_PIPE_CASE(kFp8G128Row)
    RMSQ_AR_PIPE_CASE(kFp8G128Col)
    RMSQ_AR_PIPE_CASE(kFp8G64Row)
    RMSQ_AR_PIPE_CASE(kFp8G64Col)
    RMSQ_AR_PIPE_CASE(kNvfp4)
#undef RMSQ_AR_PIPE_CASE
    default: return nullptr;
    }
}

// Launch shape of the pipelined all-reduce kernel: two chunks per thread (four
// above hidden 8192, so that a row needs at most 512 threads), a stage of
// n_ranks partial rows plus the residual row, two stages when they fit the
// ring budget, else one; the tuning's chunks per thread and stages when set.
// *ok = false when not even one stage fits (the direct kernel is used).
inline PipePlan ar_pipe_plan(const RowArgs& a, bool res, int n_ranks, bool* ok) {
    const PipeTuning tune = get_pipe_tuning();
    auto threads_for = [&](int j) { return ((a.chunks + 32 * j - 1) / (32 * j)) * 32; };
    PipePlan p;
    p.J = 2;
    if (tune.chunks_per_thread == 4) p.J = 4;
    while (p.J < 4 && threads_for(p.J) > kPipeMaxThreads) p.J *= 2;
    p.threads = threads_for(p.J);
    const int stage_bytes = a.chunks * 16 * (n_ranks + (res ? 1 : 0));
    p.stages = 2 * stage_bytes <= kPipeSmemBudget ? 2 : 1;
    if (tune.stages >= 1 && tune.stages <= kMaxStages && tune.stages * stage_bytes <= kPipeSmemBudget)
        p.stages = tune.stages;
    p.smem = p.stages * stage_bytes + co_weight_smem_bytes(p.J, p.threads * p.J);
    *ok = threads_for(p.J) <= kPipeMaxThreads && stage_bytes <= kPipeSmemBudget;
    return p;
}

// The pipelined all-reduce kernel serves up to this many ranks (measured on
// GB300, 2048-4096 rows of hidden 4096 / 7168, FP8 static): with 2 ranks
// 17.8 -> 14.9 us (hidden 4096) and 37.7 -> 25.9 us (hidden 7168), still
// ahead at 4; from 5 ranks on the direct kernel, whose many partial-row loads
// per thread are in flight at once, is faster (96-101 % of the copy peak at 8
// ranks) than a ring whose stages of 6-9 rows leave room for few CTAs.
constexpr int kArPipeMaxRanks = 4;

template <class E>
cudaError_t launch_allreduce_rows_t(const LaunchArgs& la, const void* const* partials, int n_ranks,
                                    cudaStream_t stream) {
    RowArgs a = make_row_args(la);
    ArRanks rk = {};
    rk.n = n_ranks;
    for (int r = 0; r < n_ranks; ++r) rk.part[r] = static_cast<const uint4*>(partials[r]);
    const bool res = la.res != nullptr;
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (err != cudaSuccess) return err;
    if (a.n >= kPipeMinRowsPerSm * sms && n_ranks <= kArPipeMaxRanks) {
        bool ok = false;
        const PipePlan p = ar_pipe_plan(a, res, n_ranks, &ok);
        if (ok) {
            const void* fn = pick_ar_pipe<E>(la.mode, res, p.J);
            if (!fn) return cudaErrorInvalidValue;
            int grid = 0;
            err = pipe_grid(fn, p, a.n, &grid);
            if (err != cudaSuccess) return err;
            int st = p.stages;
            void* params[] = {&a, &st, &rk};
            return launch_kernel(fn, dim3(grid), dim3(p.threads), params, p.smem, stream);
        }
    }
    a.pair = false;
    const int J = a.chunks <= 1024 ? 1 : 2;
    const int threads = ((a.chunks + J - 1) / J + 31) / 32 * 32;
    const void* fn = pick_ar_kernel<E>(la.mode, res, J);
    if (!fn) return cudaErrorInvalidValue;
    void* params[] = {&a, &rk};
    return launch_kernel(fn, dim3(a.n), dim3(threads), params, 0, stream);
}

cudaError_t launch_allreduce_rows(const LaunchArgs& la, const void* const* partials, int n_ranks, bool fp16,
                                  cudaStream_t stream) {
    if (n_ranks < 1 || n_ranks > kMaxArRanks) return cudaErrorInvalidValue;
    return fp16 ? launch_allreduce_rows_t<Fp16T>(la, partials, n_ranks, stream)
                : launch_allreduce_rows_t<Bf16T>(la, partials, n_ranks, stream);
}

cudaError_t take_pipe_fault_ar(unsigned int* out) { return take_pipe_fault(out); }

}  // namespace rmsq

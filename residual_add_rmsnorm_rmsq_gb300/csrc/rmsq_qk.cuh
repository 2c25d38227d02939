// QK-norm + RoPE (vLLM docs "Fusion torch.compile passes", section "QK Norm +
// RoPE (enable_qk_norm_rope_fusion)": split QKV, per-head RMSNorm of Q and K,
// rotary position embedding, in one kernel), in place on qkv.
//
// A head of D elements is spread over LPH = D / 16 lanes; lane g of the head
// holds two 8-element blocks, elements 8g .. 8g+7 (its "low" block) and
// D/2 + 8g .. D/2 + 8g + 7 (its "high" block).  With that layout
//  - the head's sum of squares is the canonical pairwise tree: the 8-element
//    trees of both blocks in the lane, the xor butterfly over the head's
//    lanes for the low and the high half separately, and at the root the
//    low half plus the high half;
//  - every RoPE pair is inside one lane: NeoX pairs element i with i + D/2
//    (the same position of the two blocks, angle 8g + k), GPT-J pairs 2i
//    with 2i + 1 (neighbours in a block, angle 4g + m in the low block,
//    D/4 + 4g + m in the high one), so the rotation needs no shuffles;
//  - a warp's accesses are 16-byte pieces at a 16-byte stride (coalesced in
//    global memory, free of bank conflicts in shared memory).
// The norm is the norm op's (inv = 1 / sqrt(S / D + eps), y = (x * inv) * w,
// fp32).  RoPE takes cos / sin from the caller's fp32 table at the token's
// position; every product and sum is rounded separately and the result is
// rounded once to the activation type.  v heads are not touched; a token
// whose position is outside [0, max_pos) is left unchanged.
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

// A lane holds 16 elements of its head (two blocks of 8); a head takes D / 16
// lanes (4, 8 or 16), so one warp works on 32 * 16 / D heads of a token
// together and shares the per-head scalar work (butterfly, square root,
// division) across them.
constexpr int kQkEpl = 16;

// Word offset, within a head, of the lane's low (p = 0) or high (p = 1)
// block: 4 words (16 bytes) each.
template <int D>
__device__ __forceinline__ int qk_block_word(int g, int p) { return p * (D / 4) + 4 * g; }

// First angle of the lane's cos / sin float4 q (q = 0, 1).
template <int D, bool NEOX>
__device__ __forceinline__ int qk_angle(int g, int q) {
    return NEOX ? 8 * g + 4 * q : q * (D / 4) + 4 * g;
}

// Angle source of the head math: the lane's cos / sin float4 q, from
// registers (warp kernel) or from the token's row in shared memory (pipelined
// kernel, read where they are used).
struct CsRegs {
    const float4 (&c)[2];
    const float4 (&s)[2];
    __device__ __forceinline__ float4 cos4(int q) const { return c[q]; }
    __device__ __forceinline__ float4 sin4(int q) const { return s[q]; }
};
template <int D, bool NEOX>
struct CsSmem {
    const float* row;   // the token's cos / sin row
    int g;
    __device__ __forceinline__ float4 cos4(int q) const {
        return *reinterpret_cast<const float4*>(row + qk_angle<D, NEOX>(g, q));
    }
    __device__ __forceinline__ float4 sin4(int q) const {
        return *reinterpret_cast<const float4*>(row + D / 2 + qk_angle<D, NEOX>(g, q));
    }
};

__device__ __forceinline__ float f4_at(const float4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One head group's arithmetic, shared by both kernels.  xw / ww: the lane's
// elements and weights as T pairs (words 0..3 the low block, 4..7 the high
// block); `cs` gives its angles.  Returns the rotated, normed elements in the
// same layout.
template <class E, int D, bool NEOX, class CS>
__device__ __forceinline__ void qk_head_math(const uint32_t (&xw)[8], const uint32_t (&ww)[8], const CS& cs,
                                             float eps, float inv_d, uint32_t (&ow)[8]) {
    constexpr int LPH = D / kQkEpl;
    float x[16];   // x[0..7] the low block, x[8..15] the high block
#pragma unroll
    for (int i = 0; i < 8; ++i) { x[2 * i] = E::lo(xw[i]); x[2 * i + 1] = E::hi(xw[i]); }
    // 8-element trees of both blocks, a packed pair carrying the same node
    // of the low and the high block.  Squares of bf16 / fp16 values are
    // exact in fp32, so a first-level node RN(a^2 + b^2) is one fused
    // multiply-add.
    float2 l1[2][2];   // [block][k]: first-level nodes (2k, 2k+1) of the block
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float* e = x + 8 * b + 4 * k;
            const float2 u = make_float2(e[0], e[2]), v = make_float2(e[1], e[3]);
            l1[b][k] = fma2_rn(u, u, mul2_rn(v, v));
        }
    const float2 q0 = add2_rn(make_float2(l1[0][0].x, l1[1][0].x), make_float2(l1[0][0].y, l1[1][0].y));
    const float2 q1 = add2_rn(make_float2(l1[0][1].x, l1[1][1].x), make_float2(l1[0][1].y, l1[1][1].y));
    float2 h = add2_rn(q0, q1);   // (low block, high block) sums
#pragma unroll
    for (int o = 1; o < LPH; o <<= 1)
        h = add2_rn(h, make_float2(__shfl_xor_sync(kFull, h.x, o), __shfl_xor_sync(kFull, h.y, o)));
    const float sum = __fadd_rn(h.x, h.y);   // low half + high half
    // 1 / sqrt(...) as two correctly rounded steps (the reciprocal's value is
    // the IEEE division 1 / s)
    const float inv = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(sum, inv_d), eps)));
    // y = (x * inv) * w, two elements an instruction (products only: nothing
    // to contract)
    float y[16];
    const float2 iv = make_float2(inv, inv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 t = mul2_rn(mul2_rn(make_float2(x[2 * i], x[2 * i + 1]), iv),
                                 make_float2(E::lo(ww[i]), E::hi(ww[i])));
        y[2 * i] = t.x;
        y[2 * i + 1] = t.y;
    }
    float o[16];
    if constexpr (NEOX) {
        // (a, b) = (y[k], y[8 + k]) at angle 8g + k: a c - b s, b c + a s
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 c4 = cs.cos4(q), s4 = cs.sin4(q);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int k = 4 * q + i;
                const float c = f4_at(c4, i), sn = f4_at(s4, i);
                o[k] = __fsub_rn(__fmul_rn(y[k], c), __fmul_rn(y[8 + k], sn));
                o[8 + k] = __fadd_rn(__fmul_rn(y[8 + k], c), __fmul_rn(y[k], sn));
            }
        }
    } else {
        // (a, b) = (y[8q + 2m], y[8q + 2m + 1]) at cos / sin element m of float4 q
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 c4 = cs.cos4(q), s4 = cs.sin4(q);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float c = f4_at(c4, m), sn = f4_at(s4, m);
                const float ya = y[8 * q + 2 * m], yb = y[8 * q + 2 * m + 1];
                o[8 * q + 2 * m] = __fsub_rn(__fmul_rn(ya, c), __fmul_rn(yb, sn));
                o[8 * q + 2 * m + 1] = __fadd_rn(__fmul_rn(yb, c), __fmul_rn(ya, sn));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ow[i] = E::pack(o[2 * i], o[2 * i + 1]);
}

__device__ __forceinline__ void unpack2(const uint4& a, const uint4& b, uint32_t (&w)[8]) {
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// Resident 256-thread CTAs per SM the warp kernel is compiled for (the
// register budget follows from it); compile-time tuning, results do not
// depend on it.  Tighter budgets spill and were slower on GB300.
#ifndef RMSQ_QK_MIN_BLOCKS
#define RMSQ_QK_MIN_BLOCKS 1
#endif

// Warp kernel (few tokens): each warp takes one head group of one token,
// loads straight into registers, computes and stores; warps stride over the
// n * (head groups per token) work items.
template <class E, int D, bool NEOX>
__global__ void __launch_bounds__(256, RMSQ_QK_MIN_BLOCKS) qk_norm_rope_kernel(const QkArgs a) {
    constexpr int LPH = D / kQkEpl;             // lanes per head
    constexpr int HPW = 32 / LPH;               // heads per warp
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
        uint32_t xw[8] = {}, ww[8] = {};
        uint32_t* hp = a.qkv + (int64_t)t * width_words + hd * (D / 2);
        if (live) {
            const uint32_t* wp = hd < a.nq ? a.qw : a.kw;
            unpack2(ld_act(reinterpret_cast<const uint4*>(hp + qk_block_word<D>(g, 0))),
                    ld_act(reinterpret_cast<const uint4*>(hp + qk_block_word<D>(g, 1))), xw);
            unpack2(__ldg(reinterpret_cast<const uint4*>(wp + qk_block_word<D>(g, 0))),
                    __ldg(reinterpret_cast<const uint4*>(wp + qk_block_word<D>(g, 1))), ww);
        }
        const float* row = a.cs + p * D;
        const float4 cv[2] = {__ldg(reinterpret_cast<const float4*>(row + qk_angle<D, NEOX>(g, 0))),
                              __ldg(reinterpret_cast<const float4*>(row + qk_angle<D, NEOX>(g, 1)))};
        const float4 sv[2] = {__ldg(reinterpret_cast<const float4*>(row + D / 2 + qk_angle<D, NEOX>(g, 0))),
                              __ldg(reinterpret_cast<const float4*>(row + D / 2 + qk_angle<D, NEOX>(g, 1)))};
        uint32_t ow[8];
        qk_head_math<E, D, NEOX>(xw, ww, CsRegs{cv, sv}, a.eps, a.inv_d, ow);
        if (live) {
            st_stream(reinterpret_cast<uint4*>(hp + qk_block_word<D>(g, 0)), make_uint4(ow[0], ow[1], ow[2], ow[3]));
            st_stream(reinterpret_cast<uint4*>(hp + qk_block_word<D>(g, 1)), make_uint4(ow[4], ow[5], ow[6], ow[7]));
        }
    }
}

// Pipelined form for large batches: persistent CTAs, each walking the tokens
// blockIdx.x + k * gridDim.x.  One elected thread keeps the q and k heads of
// the next `stages` tokens (contiguous in the token's row) and their cos / sin
// rows in flight as 1-D bulk asynchronous copies (TMA) into a ring of
// shared-memory stages; the warps take the token's heads HPW at a time from
// shared memory with exactly the arithmetic above and store to global
// memory.  A stage is refilled after the CTA barrier that ends its token (a
// dedicated producer warp with per-stage "empty" barriers instead measured no
// faster on GB300: the warps are bound by instruction issue, not by the
// barrier).  The token's position is read by the elected thread one refill
// ahead and handed over in shared memory (the mbarrier's arrive / wait order
// it).  Every wait is bounded; a CTA that gives up records it in the unit's
// fault flag (read by rmsq_take_fault_flags), drains its copies (bounded
// again) and returns.
constexpr int kQkMaxStages = 8;
constexpr int kQkPipeMaxThreads = 512;
// Register budget of the pipelined kernel (per thread; at most 64, so that a
// CTA of up to kQkPipeMaxThreads threads always fits an SM): 56 allows four
// of its usual 288-thread CTAs per SM (64: three) without spilling, 3-6 %
// faster on GB300; 48 spills.  Compile-time tuning, results do not depend
// on it.
#ifndef RMSQ_QK_PIPE_MAXNREG
#define RMSQ_QK_PIPE_MAXNREG 56
#endif
static_assert(RMSQ_QK_PIPE_MAXNREG <= 64, "a 512-thread CTA must fit the SM's registers");

template <class E, int D, bool NEOX>
__global__ void __maxnreg__(RMSQ_QK_PIPE_MAXNREG)
    qk_pipe_kernel(const QkArgs a, const int stages, const uint32_t stage_bytes) {
    constexpr int LPH = D / kQkEpl, HPW = 32 / LPH;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kQkMaxStages];
    __shared__ int64_t s_pos[kQkMaxStages];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int g = lane % LPH, r = lane / LPH;
    const int heads = a.nq + a.nkv;
    const int chunks = (heads + HPW - 1) / HPW;
    const int width_words = (heads + a.nkv) * D / 2;
    const uint32_t head_bytes = static_cast<uint32_t>(heads) * D * 2;   // q and k heads of a token
    const int G = gridDim.x;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    allow_dependents();
    grid_dependency_wait();
    __syncthreads();

    // Thread 0: start the copies of token k (position p) into stage s.
    uint64_t pol_first = 0, pol_keep = 0;
    auto issue = [&](int k, int s, int64_t p) {
        const int t = blockIdx.x + k * G;
        unsigned char* dst = ring + (size_t)s * stage_bytes;
        const bool valid = p >= 0 && p < a.max_pos;
        s_pos[s] = p;
        mbar_arrive_expect_tx(&full[s], head_bytes + (valid ? D * 4u : 0u));
        bulk_g2s(dst, a.qkv + (int64_t)t * width_words, head_bytes, &full[s], pol_first);
        if (valid) bulk_g2s(dst + head_bytes, a.cs + p * D, D * 4u, &full[s], pol_keep);
    };
    int64_t p_next = -1;   // thread 0: position of the next token to issue
    if (tid == 0) {
        pol_first = l2_policy_evict_first();
        pol_keep = l2_policy_evict_normal();
        int64_t pp[kQkMaxStages];
#pragma unroll
        for (int k = 0; k < kQkMaxStages; ++k) {
            const int t = blockIdx.x + k * G;
            pp[k] = (k < stages && t < a.n) ? __ldg(a.pos + t) : -1;
        }
#pragma unroll
        for (int k = 0; k < kQkMaxStages; ++k)
            if (k < stages && blockIdx.x + k * G < a.n) issue(k, k, pp[k]);
        const int t = blockIdx.x + stages * G;
        if (t < a.n) p_next = __ldg(a.pos + t);
    }

    // The weight words of the warp's head group (the same for every token
    // while the warp has one group; reloaded per token otherwise).
    uint32_t ww[8] = {};
    auto load_w = [&](int c) {
        const int hd = c * HPW + r;
        if (hd < heads) {
            const uint32_t* wp = hd < a.nq ? a.qw : a.kw;
            unpack2(__ldg(reinterpret_cast<const uint4*>(wp + qk_block_word<D>(g, 0))),
                    __ldg(reinterpret_cast<const uint4*>(wp + qk_block_word<D>(g, 1))), ww);
        }
    };
    load_w(warp);

    int k = 0, s = 0;
    uint32_t parity = 0;   // stage s and its phase, advanced per token (no division)
    bool faulted = false;
    for (;; ++k) {
        const int t = blockIdx.x + k * G;
        if (t >= a.n) break;
        // one answer per warp: the head math below shuffles across all lanes
        const bool ok = __all_sync(kFull, mbar_wait_bounded(&full[s], parity));
        const int64_t p = s_pos[s];
        if (ok && p >= 0 && p < a.max_pos) {
            const unsigned char* st = ring + (size_t)s * stage_bytes;
            const CsSmem<D, NEOX> cs{reinterpret_cast<const float*>(st + head_bytes), g};
            for (int c = warp; c < chunks; c += nwarps) {
                const int hd = c * HPW + r;
                const bool live = hd < heads;
                if (c != warp) load_w(c);   // more head groups than warps
                uint32_t xw[8] = {};
                if (live) {
                    const uint32_t* sp = reinterpret_cast<const uint32_t*>(st) + hd * (D / 2);
                    unpack2(*reinterpret_cast<const uint4*>(sp + qk_block_word<D>(g, 0)),
                            *reinterpret_cast<const uint4*>(sp + qk_block_word<D>(g, 1)), xw);
                }
                uint32_t ow[8];
                qk_head_math<E, D, NEOX>(xw, ww, cs, a.eps, a.inv_d, ow);
                if (chunks > nwarps && c + nwarps >= chunks) load_w(warp);   // back to the first group
                if (live) {
                    uint32_t* hp = a.qkv + (int64_t)t * width_words + hd * (D / 2);
                    st_stream(reinterpret_cast<uint4*>(hp + qk_block_word<D>(g, 0)),
                              make_uint4(ow[0], ow[1], ow[2], ow[3]));
                    st_stream(reinterpret_cast<uint4*>(hp + qk_block_word<D>(g, 1)),
                              make_uint4(ow[4], ow[5], ow[6], ow[7]));
                }
            }
        }
        // Every read of stage s is done once all threads are past this barrier.
        if (__syncthreads_or(!ok)) {
            faulted = true;
            break;
        }
        if (tid == 0 && blockIdx.x + (k + stages) * G < a.n) {
            issue(k + stages, s, p_next);
            const int tn = blockIdx.x + (k + stages + 1) * G;
            if (tn < a.n) p_next = __ldg(a.pos + tn);
        }
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
    if (faulted && tid == 0) {
        atomicOr(&g_pipe_fault, 1u);
        for (int kk = k; kk < k + stages; ++kk) {
            if (blockIdx.x + kk * G >= a.n) break;
            mbar_wait_bounded(&full[kk % stages], static_cast<uint32_t>(kk / stages) & 1u);
        }
    }
}

// Ring stage of the pipelined form: the q and k heads of a token and its
// cos / sin row, rounded up to 128 bytes.
inline uint32_t qk_stage_bytes(int heads, int head_dim) {
    return (static_cast<uint32_t>(heads) * head_dim * 2 + head_dim * 4 + 127u) / 128u * 128u;
}

// Stages of the ring: about 24 KB of copies per CTA, 2 to kQkMaxStages
// (deeper rings measured no faster on GB300: the kernel is bound by its
// per-token instruction chain, not by the bytes in flight).
inline int qk_stages(uint32_t stage_bytes) {
    int s = static_cast<int>((24u * 1024u) / stage_bytes);
    if (s < 2) s = 2;
    if (s > kQkMaxStages) s = kQkMaxStages;
    while (s > 2 && static_cast<uint32_t>(s) * stage_bytes > static_cast<uint32_t>(kPipeSmemBudget)) --s;
    return s;
}

// Pipelined when asked for (or, for AUTO, from eight tokens per SM up: below
// that the warp kernel's lower latency wins on GB300) and two stages fit the
// shared-memory budget; otherwise the warp kernel.
template <class E>
cudaError_t launch_qk(const QkArgs& a, int head_dim, bool neox, int variant, cudaStream_t stream) {
    cudaError_t err = cudaSuccess;
    const int sms = sm_count(&err);
    if (err != cudaSuccess) return err;
    const int hpw = 32 * kQkEpl / head_dim;
    const int heads = a.nq + a.nkv;
    const int chunks = (heads + hpw - 1) / hpw;
    const uint32_t stage_bytes = qk_stage_bytes(heads, head_dim);
    const bool fits = 2u * stage_bytes <= static_cast<uint32_t>(kPipeSmemBudget);
    const bool pipe = fits && variant != kVariantDirect && (variant == kVariantPipelined || a.n >= 8 * sms);
    QkArgs args = a;
    if (pipe) {
        const void* fn = nullptr;
        switch (head_dim) {
        case 64: fn = neox ? (const void*)&qk_pipe_kernel<E, 64, true> : (const void*)&qk_pipe_kernel<E, 64, false>; break;
        case 128: fn = neox ? (const void*)&qk_pipe_kernel<E, 128, true> : (const void*)&qk_pipe_kernel<E, 128, false>; break;
        case 256: fn = neox ? (const void*)&qk_pipe_kernel<E, 256, true> : (const void*)&qk_pipe_kernel<E, 256, false>; break;
        default: return cudaErrorInvalidValue;
        }
        // warps: the token's head groups spread evenly, at most 16
        const int passes = (chunks + 15) / 16;
        const int warps = (chunks + passes - 1) / passes;
        const int threads = warps * 32;
        int stages = qk_stages(stage_bytes);
        const PipeTuning tune = get_pipe_tuning();
        if (tune.stages >= 2 && tune.stages <= kQkMaxStages &&
            static_cast<uint32_t>(tune.stages) * stage_bytes <= static_cast<uint32_t>(kPipeSmemBudget))
            stages = tune.stages;
        const int smem = stages * static_cast<int>(stage_bytes);
        int per_sm = pipe_blocks_per_sm(fn, threads, smem, &err);
        if (err != cudaSuccess) return err;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        if (tune.ctas_per_sm >= 1 && tune.ctas_per_sm < per_sm) per_sm = tune.ctas_per_sm;
        const int grid = a.n < per_sm * sms ? a.n : per_sm * sms;
        uint32_t sb = stage_bytes;
        void* params[] = {&args, &stages, &sb};
        return launch_kernel(fn, dim3(grid), dim3(threads), params, smem, stream);
    }
    const void* fn = nullptr;
    switch (head_dim) {
    case 64: fn = neox ? (const void*)&qk_norm_rope_kernel<E, 64, true> : (const void*)&qk_norm_rope_kernel<E, 64, false>; break;
    case 128: fn = neox ? (const void*)&qk_norm_rope_kernel<E, 128, true> : (const void*)&qk_norm_rope_kernel<E, 128, false>; break;
    case 256: fn = neox ? (const void*)&qk_norm_rope_kernel<E, 256, true> : (const void*)&qk_norm_rope_kernel<E, 256, false>; break;
    default: return cudaErrorInvalidValue;
    }
    const int64_t warps = (int64_t)a.n * chunks;
    int64_t grid = (warps + 7) / 8;
    if (grid > (int64_t)sms * 32) grid = (int64_t)sms * 32;
    void* params[] = {&args};
    return launch_kernel(fn, dim3((unsigned)grid), dim3(256), params, 0, stream);
}

}  // namespace rmsq

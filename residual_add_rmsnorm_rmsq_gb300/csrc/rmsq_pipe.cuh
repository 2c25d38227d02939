// Pipelined row kernel: persistent CTAs, each walking the rows blockIdx.x,
// blockIdx.x + gridDim.x, ...; the x and residual rows of the next `stages`
// rows are in flight as bulk asynchronous copies (TMA, 1-D) into a ring of
// shared-memory stages while the current row is computed.  One elected
// thread issues the copies; a stage is refilled right after the CTA barrier
// that follows its last shared-memory read.
//
// Data-to-thread mapping (coalesced): lane l of warp w holds the chunks
// c = (w * J + j) * 32 + l, j = 0 .. J-1, of a row (a chunk is 16 bytes, 8
// elements).  A warp's j-th access covers 512 contiguous bytes, so the ring
// reads are free of bank conflicts and the residual and code stores are
// fully coalesced.  The canonical pairwise tree of the sum of squares maps
// onto it without reordering: the tree over a chunk's 8 elements, an xor
// butterfly over the lanes for each j (bits 0..4 of the chunk index), the
// tree over j (the next log2 J bits), then the tree over the warps' sums
// (zero-padded, exact).
//
// Per row the arithmetic is the direct kernel's (rmsq_rowmath.cuh): the
// canonical tree, correctly rounded inverse RMS, y = (h * inv) * w in fp32,
// then the quantisation mode; only the order in which the threads visit the
// elements differs, never a rounding.
//
// Every wait on a stage is bounded (mbar_wait_bounded).  If one ever gives up,
// the CTA records it in `fault`, drains the copies it still has in flight
// (again bounded) and returns.
#pragma once

#include "rmsq_launch.h"
#include "rmsq_rowmath.cuh"

namespace rmsq {

// The ranks' partial-sum buffers of the all-reduce variant, passed by value
// in the kernel parameters.
struct ArRanks {
    const uint4* part[kMaxArRanks];
    int n;
};

// x = T(sum over ranks of fp32(partial)) for one chunk whose n partials sit
// `stride` chunks apart in shared memory: rank order, one rounding at the
// end (the all-reduce's reduction; the direct all-reduce kernel adds the same
// values in the same order).
template <class E>
__device__ __forceinline__ uint4 ar_chunk_sum(const uint4* p, int stride, int n) {
    const uint4 v0 = p[0];
    const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
    float acc[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) { acc[2 * k] = E::lo(w0[k]); acc[2 * k + 1] = E::hi(w0[k]); }
    for (int r = 1; r < n; ++r) {
        const uint4 v = p[(size_t)r * stride];
        const uint32_t wr[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 t = add2_rn(make_float2(acc[2 * k], acc[2 * k + 1]), make_float2(E::lo(wr[k]), E::hi(wr[k])));
            acc[2 * k] = t.x;
            acc[2 * k + 1] = t.y;
        }
    }
    return make_uint4(E::pack(acc[0], acc[1]), E::pack(acc[2], acc[3]), E::pack(acc[4], acc[5]),
                      E::pack(acc[6], acc[7]));
}

constexpr int kMaxStages = 8;
constexpr int kPipeMaxThreads = 512;

// The warp's node of the canonical tree over its 32 * J chunks (the same
// value in every lane): leaf trees of the lane's chunks, the lane butterfly
// of each j (two j at a time in packed pairs), then the tree over j.
template <int J>
__device__ __forceinline__ float co_warp_sum(const float (&h)[J][8]) {
    if constexpr (J == 1) {
        return warp_tree_sum(leaf8_sumsq(h[0]));
    } else {
        float p[J];
#pragma unroll
        for (int j = 0; j < J; j += 2) {
            float2 v = leaf8_sumsq2(h[j], h[j + 1]);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1)
                v = add2_rn(v, make_float2(__shfl_xor_sync(kFull, v.x, o), __shfl_xor_sync(kFull, v.y, o)));
            p[j] = v.x;
            p[j + 1] = v.y;
        }
#pragma unroll
        for (int len = J; len > 1; len >>= 1)
#pragma unroll
            for (int i = 0; i < len / 2; ++i) p[i] = __fadd_rn(p[2 * i], p[2 * i + 1]);
        return p[0];
    }
}

// Weights of the thread's chunks, loaded once per CTA and widened to fp32:
// in registers for one or two chunks per thread; for more, in the CTA's
// shared memory (where the registers serve occupancy better), each thread's
// own chunks in a lane-interleaved layout (two float4 per chunk, the warp's
// 32 lanes side by side: conflict-free 16-byte reads).  A thread reads back
// only what it wrote, so no barrier is needed; the reads are volatile so that
// the compiler keeps them in the row loop instead of hoisting them into
// registers.
// Compile-time tuning (results do not depend on it): 0 keeps the weights of
// four or eight chunks per thread packed in registers instead.
#ifndef RMSQ_PIPE_WSMEM
#define RMSQ_PIPE_WSMEM 1
#endif

template <class E, int J>
struct CoWeights {
    static constexpr bool kSmem = J >= 4 && RMSQ_PIPE_WSMEM;
    static constexpr bool kPacked = J >= 4 && !RMSQ_PIPE_WSMEM;
    float f[(kSmem || kPacked) ? 1 : J][8];
    uint32_t pk[kPacked ? J : 1][4];
    float4* wsm;   // kSmem: this thread's first float4; chunk j at +(2 j) * 32 and +(2 j + 1) * 32

    __device__ __forceinline__ void load(const uint4* w, int c0, int chunks, float4* smem_w, int warp, int lane) {
        wsm = smem_w + (size_t)warp * J * 64 + lane;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int c = c0 + 32 * j;
            const uint4 v = c < chunks ? ld_weight(w + c) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
            float t[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) { t[2 * k] = E::lo(ws[k]); t[2 * k + 1] = E::hi(ws[k]); }
            if constexpr (kSmem) {
                wsm[(2 * j) * 32] = make_float4(t[0], t[1], t[2], t[3]);
                wsm[(2 * j + 1) * 32] = make_float4(t[4], t[5], t[6], t[7]);
            } else if constexpr (kPacked) {
#pragma unroll
                for (int k = 0; k < 4; ++k) pk[j][k] = ws[k];
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) f[j][k] = t[k];
            }
        }
    }
    // The eight weights of chunk j.
    __device__ __forceinline__ void get(int j, float (&o)[8]) const {
        if constexpr (kSmem) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float4* p = wsm + (2 * j + hf) * 32;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(o[4 * hf]), "=f"(o[4 * hf + 1]), "=f"(o[4 * hf + 2]), "=f"(o[4 * hf + 3])
                             : "r"(smem_u32(p)));
            }
        } else if constexpr (kPacked) {
            // through an empty volatile asm, so that the widening stays in the
            // row loop instead of being hoisted into registers
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t v = pk[j][k];
                asm volatile("" : "+r"(v));
                o[2 * k] = E::lo(v);
                o[2 * k + 1] = E::hi(v);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = f[j][k];
        }
    }
};

// Shared-memory bytes of the weights of a pipelined launch (none for one or
// two chunks per thread).
__host__ __device__ constexpr int co_weight_smem_bytes(int J, int chunks_covered) {
    return (J >= 4 && RMSQ_PIPE_WSMEM) ? chunks_covered * 32 : 0;
}

// y = (h * inv) * w in place over h, in packed pairs (element k of chunks j
// and j + 1; elements k and k + 1 of the one chunk when J == 1).
template <class E, int J>
__device__ __forceinline__ void co_y(float (&h)[J][8], const CoWeights<E, J>& w, float inv) {
    const float2 iv = make_float2(inv, inv);
    if constexpr (J == 1) {
        float wf[8];
        w.get(0, wf);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float2 t = mul2_rn(mul2_rn(make_float2(h[0][k], h[0][k + 1]), iv), make_float2(wf[k], wf[k + 1]));
            h[0][k] = t.x;
            h[0][k + 1] = t.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < J; j += 2) {
            float wa[8], wb[8];
            w.get(j, wa);
            w.get(j + 1, wb);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 t = mul2_rn(mul2_rn(make_float2(h[j][k], h[j + 1][k]), iv), make_float2(wa[k], wb[k]));
                h[j][k] = t.x;
                h[j + 1][k] = t.y;
            }
        }
    }
}

// E4M3 codes of the thread's chunks, chunk j divided by s[j], stored as 8
// bytes per chunk (a warp's j-th store is 256 contiguous bytes).
template <int J>
__device__ __forceinline__ void co_store_fp8(const RowArgs& a, int row, const float (&y)[J][8], const float (&s)[J],
                                             const Fp8Recips (&rc)[J], int c0) {
    uint2* qrow = reinterpret_cast<uint2*>(a.q + (int64_t)row * a.hidden);
    uint2 codes[J];
    if constexpr (J == 1) {
        codes[0] = fp8_chunk(y[0], s[0], rc[0]);
    } else {
#pragma unroll
        for (int j = 0; j < J; j += 2) fp8_chunk2s(y[j], y[j + 1], s[j], s[j + 1], rc[j], rc[j + 1], codes[j], codes[j + 1]);
    }
#pragma unroll
    for (int j = 0; j < J; ++j)
        if (c0 + 32 * j < a.chunks) st_stream(qrow + c0 + 32 * j, codes[j]);
}

// AR: x is the all-reduce of the ranks' partial rows (rk), each copied into
// the stage beside the residual row.
template <class E, int MODE, bool RES, int J, bool AR = false>
__device__ __forceinline__ void pipe_body(const RowArgs& a, const int stages, unsigned int* fault,
                                          const ArRanks* rk = nullptr) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ __align__(16) float s_sum[2][32];
    __shared__ float s_max[32];
    __shared__ float s_rtab[MODE == kNvfp4 ? 128 : 1];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int c0 = warp * J * 32 + lane;   // the thread's first chunk; the others follow at strides of 32
    const int G = gridDim.x;
    const uint32_t row_bytes = static_cast<uint32_t>(a.chunks) * 16u;
    const int nsrc = AR ? rk->n : 1;   // rows that make up x
    // one row of x (or of each rank's partial) (+ residual)
    const uint32_t stage_bytes = static_cast<uint32_t>(nsrc + (RES ? 1 : 0)) * row_bytes;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    // Slots of absent warps read as 0, in both halves of the double buffer,
    // whatever the CTA size.
    for (int i = tid; i < 64; i += blockDim.x)
        if ((i & 31) >= nwarps) (&s_sum[0][0])[i] = 0.0f;
    allow_dependents();
    grid_dependency_wait();
    __syncthreads();

    // Thread 0: start the copies of `row` into stage s.  The first pass of
    // the data-derived NVFP4 scale is followed by a pass that reads h again:
    // without a residual h is x, kept in L2 at normal priority.
    constexpr bool KEEP = MODE == kNormAmax;
    uint64_t policy = 0;
    auto issue = [&](int row, int s) {
        unsigned char* dst = ring + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        if constexpr (AR) {
            for (int r = 0; r < nsrc; ++r)
                bulk_g2s(dst + (size_t)r * row_bytes, rk->part[r] + (int64_t)row * a.chunks, row_bytes, &full[s],
                         policy);
        } else {
            bulk_g2s(dst, a.x + (int64_t)row * a.chunks, row_bytes, &full[s], policy);
        }
        if constexpr (RES)
            bulk_g2s(dst + (size_t)nsrc * row_bytes, a.res + (int64_t)row * a.chunks, row_bytes, &full[s], policy);
    };
    if (tid == 0) {
        policy = (KEEP && !RES) ? l2_policy_evict_normal() : l2_policy_evict_first();
        for (int k = 0; k < stages; ++k) {
            if (blockIdx.x + k * G >= a.n) break;
            issue(blockIdx.x + k * G, k);
        }
    }

    CoWeights<E, J> wts;
    wts.load(a.w, c0, a.chunks, reinterpret_cast<float4*>(ring + (size_t)stages * stage_bytes), warp, lane);
    const float sin = ModeTraits<MODE>::needs_scale_in ? __ldg(a.scale_in) : 0.0f;
    if constexpr (MODE == kNvfp4) fill_nvfp4_rtab(s_rtab, sin);   // ordered by the first row's barrier
    Fp8Recips rc_static = {0.0f, 0.0f};
    if constexpr (MODE == kFp8Static) rc_static = fp8_recips(sin);

    int s = 0, buf = 0;
    uint32_t parity = 0;
    int row = blockIdx.x;
    bool faulted = false;
    float run_max = 0.0f;
    for (; row < a.n; row += G) {
        const bool ok = mbar_wait_bounded(&full[s], parity);

        // h = T(x + r) (h = x without a residual), the write-back, widened.
        float h[J][8];
        {
            const uint4* sx = reinterpret_cast<const uint4*>(ring + (size_t)s * stage_bytes);
            uint4* ro = a.res_out + (int64_t)row * a.chunks;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int c = c0 + 32 * j;
                uint32_t hw[4] = {0u, 0u, 0u, 0u};
                if (ok && c < a.chunks) {
                    uint4 xv;
                    if constexpr (AR) xv = ar_chunk_sum<E>(sx + c, a.chunks, nsrc);
                    else xv = sx[c];
                    hw[0] = xv.x; hw[1] = xv.y; hw[2] = xv.z; hw[3] = xv.w;
                    if constexpr (RES) {
                        const uint4 rv = sx[(size_t)nsrc * a.chunks + c];
                        const uint32_t rs[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) hw[k] = E::add2(hw[k], rs[k]);
                        const uint4 v = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        if constexpr (KEEP) st_keep(ro + c, v);
                        else st_stream(ro + c, v);
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) { h[j][2 * k] = E::lo(hw[k]); h[j][2 * k + 1] = E::hi(hw[k]); }
            }
        }
        const float wsum = co_warp_sum<J>(h);
        if (lane == 0) s_sum[buf][warp] = wsum;
        // All reads of stage s are done once every thread is past this barrier.
        if (__syncthreads_or(!ok)) {
            faulted = true;
            break;
        }
        if (tid == 0 && row + stages * G < a.n) issue(row + stages * G, s);

        const float inv = inv_rms(warp_slots_tree_sum<kPipeMaxThreads / 32>(s_sum[buf], nwarps), a);
        co_y<E, J>(h, wts, inv);   // h now holds y

        if constexpr (MODE == kNormAmax) {
#pragma unroll
            for (int j = 0; j < J; ++j) run_max = max_abs8(run_max, h[j]);
            if (tid == 0) static_cast<float*>(a.scales)[kWsInvOffset + row] = inv;
        } else if constexpr (MODE == kNormOnly) {
            uint4* yrow = reinterpret_cast<uint4*>(a.q) + (int64_t)row * a.chunks;
#pragma unroll
            for (int j = 0; j < J; ++j)
                if (c0 + 32 * j < a.chunks)
                    st_stream(yrow + c0 + 32 * j, make_uint4(E::pack(h[j][0], h[j][1]), E::pack(h[j][2], h[j][3]),
                                                             E::pack(h[j][4], h[j][5]), E::pack(h[j][6], h[j][7])));
        } else if constexpr (MODE == kFp8Static) {
            float sv[J];
            Fp8Recips rc[J];
#pragma unroll
            for (int j = 0; j < J; ++j) { sv[j] = sin; rc[j] = rc_static; }
            co_store_fp8<J>(a, row, h, sv, rc, c0);
        } else if constexpr (MODE == kFp8PerToken) {
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j) m = max_abs8(m, h[j]);
            m = warp_max_nonneg(m);
            if (lane == 0) s_max[warp] = m;
            __syncthreads();
            m = warp_max_nonneg(lane < nwarps ? s_max[lane] : 0.0f);
            float sc = fmaxf(__fdiv_rn(m, 448.0f), 1e-12f);
            if (a.e8m0) sc = pow2_ceil(sc);
            if (tid == 0) store_scale(a, row, sc);
            const Fp8Recips r1 = fp8_recips_dyn(sc);
            float sv[J];
            Fp8Recips rc[J];
#pragma unroll
            for (int j = 0; j < J; ++j) { sv[j] = sc; rc[j] = r1; }
            co_store_fp8<J>(a, row, h, sv, rc, c0);
        } else if constexpr (MODE == kNvfp4) {
            // 16-element blocks are chunk pairs (2m, 2m + 1): lane pairs.
            const float gs = sin;
            uint8_t* bsc = static_cast<uint8_t*>(a.scales) + (int64_t)row * (a.hidden / 16);
            uint32_t* qrow = reinterpret_cast<uint32_t*>(a.q + (int64_t)row * (a.hidden / 2));
            float r[J];
            uint32_t sb[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                float m = max_abs8(0.0f, h[j]);
                m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
                sb[j] = e4m3x2(__fmul_rn(__fdiv_rn(m, 6.0f), gs), 0.0f) & 0xffu;
                r[j] = s_rtab[sb[j]];   // gs / decode(sb), 0 for a zero block scale
            }
#pragma unroll
            for (int j = 0; j < J; j += (J == 1 ? 1 : 2)) {
                uint32_t codes[2];
                if constexpr (J == 1) {
                    float v[8];
#pragma unroll
                    for (int k = 0; k < 8; k += 2) {
                        const float2 t = mul2_rn(make_float2(h[0][k], h[0][k + 1]), make_float2(r[0], r[0]));
                        v[k] = t.x; v[k + 1] = t.y;
                    }
                    codes[0] = e2m1x8(v);
                } else {
                    float v0[8], v1[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float2 t = mul2_rn(make_float2(h[j][k], h[j + 1][k]), make_float2(r[j], r[j + 1]));
                        v0[k] = t.x; v1[k] = t.y;
                    }
                    codes[0] = e2m1x8(v0);
                    codes[1] = e2m1x8(v1);
                }
#pragma unroll
                for (int u = 0; u < (J == 1 ? 1 : 2); ++u) {
                    const int c = c0 + 32 * (j + u);
                    if (c < a.chunks) {
                        st_stream(qrow + c, codes[u]);
                        if ((lane & 1) == 0) bsc[c >> 1] = (uint8_t)sb[j + u];
                    }
                }
            }
        } else {
            // FP8 per group of G contiguous elements: G / 8 lanes of one j.
            constexpr int GL = ModeTraits<MODE>::group / 8;
            float sv[J];
            Fp8Recips rc[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const float m = lanes_max<GL>(max_abs8(0.0f, h[j]));
                float sc = fmaxf(__fdiv_rn(m, 448.0f), 1e-12f);
                if (a.e8m0) sc = pow2_ceil(sc);
                sv[j] = sc;
                rc[j] = fp8_recips_dyn(sc);
                const int c = c0 + 32 * j;
                if (c < a.chunks && (lane % GL) == 0) {
                    const int g = c / GL;
                    if constexpr (ModeTraits<MODE>::col) store_scale(a, (int64_t)g * a.col_stride + row, sc);
                    else store_scale(a, (int64_t)row * (a.hidden / ModeTraits<MODE>::group) + g, sc);
                }
            }
            co_store_fp8<J>(a, row, h, sv, rc, c0);
        }

        buf ^= 1;
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
    if constexpr (MODE == kNormAmax) flush_amax(a, run_max, s_max, tid, nwarps);

    if (faulted && tid == 0) {
        atomicOr(fault, 1u);
        // Copies issued for this row and the next stages - 1 rows may still be in flight.
        for (int i = 0; i < stages; ++i) {
            if (row + i * G >= a.n) break;
            int ss = s + i;
            uint32_t pp = parity;
            if (ss >= stages) {
                ss -= stages;
                pp ^= 1u;
            }
            mbar_wait_bounded(&full[ss], pp);
        }
    }
}

}  // namespace rmsq

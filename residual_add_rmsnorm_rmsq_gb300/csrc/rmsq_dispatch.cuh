// Picks the row-kernel instantiation for (mode, residual, chunks per thread)
// and launches it: one CTA per row, ceil(hidden / 8 / J) threads rounded up
// to whole warps.
#pragma once

#include "rmsq_launch.h"
#include "rmsq_rows.cuh"

namespace rmsq {

template <class E, int MODE, bool RES>
const void* pick_j(int J) {
    if (J == 1) return reinterpret_cast<const void*>(&rows_kernel<E, MODE, RES, 1>);
    return reinterpret_cast<const void*>(&rows_kernel<E, MODE, RES, 2>);
}

template <class E, int MODE>
const void* pick_res(bool res, int J) {
    return res ? pick_j<E, MODE, true>(J) : pick_j<E, MODE, false>(J);
}

template <class E>
const void* pick_kernel(int mode, bool res, int J) {
    switch (mode) {
    case kFp8Static: return pick_res<E, kFp8Static>(res, J);
    case kFp8PerToken: return pick_res<E, kFp8PerToken>(res, J);
    case kFp8G128Row: return pick_res<E, kFp8G128Row>(res, J);
    case kFp8G128Col: return pick_res<E, kFp8G128Col>(res, J);
    case kFp8G64Row: return pick_res<E, kFp8G64Row>(res, J);
    case kFp8G64Col: return pick_res<E, kFp8G64Col>(res, J);
    case kNvfp4: return pick_res<E, kNvfp4>(res, J);
    default: return nullptr;
    }
}

template <class E>
cudaError_t launch_rows(const LaunchArgs& la, cudaStream_t stream) {
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
    const int J = a.chunks <= 1024 ? 1 : 2;
    const int threads = ((a.chunks + J - 1) / J + 31) / 32 * 32;
    const void* fn = pick_kernel<E>(la.mode, la.res != nullptr, J);
    if (!fn) return cudaErrorInvalidValue;
    void* params[] = {&a};
    return cudaLaunchKernel(fn, dim3(a.n), dim3(threads), params, 0, stream);
}

}  // namespace rmsq

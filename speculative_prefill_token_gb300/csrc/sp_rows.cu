// Sparse-prefill consumer of the SpecPrefill path ("SpecPrefill —
// Implementation Guide", §How It Works / Sparse Prefill): the target
// prefills only the kept tokens, each at its original position. Two gathers
// feed it from the kept list that the scoring path leaves on the device:
//  - gather_tokens: the kept tokens' ids, in kept order, for the target's
//    batch (the positions are the scoring path's kept_pos already);
//  - gather_rows: the kept tokens' rows of a token-major cache tensor
//    (keys or values built from the draft), packed densely.
//
// The sliding-window scoring of the pages' tool merges per-window
// importance the same way (merge_windows_kernel).
//
// All are HBM-bound copies. gather_rows gives every (layer, kept row) to
// one warp, which issues all of its 16-byte streaming loads for up to 4
// vectors per lane before the stores, so that one warp keeps a whole row
// of a typical cache in flight; a grid of 8 CTAs per SM strides over the
// rows. The kept count is read on the device.
#include <cuda_runtime.h>

#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {
namespace {

constexpr int kRowsThreads = 256;
constexpr int kRowsWarps = kRowsThreads / 32;
constexpr int kRowsUnroll = 4;
constexpr int kRowsCtasPerSm = 8;

struct RowsArgs {
    const int32_t* kept_idx;
    const int32_t* n_kept;
    const uint16_t* src;
    uint16_t* dst;
    int64_t ntot, dst_rows, ks_layer, ks_token, ks_head;  // element strides of src
    int ly, hk, d;
};

__device__ __forceinline__ int64_t clamp_kept(const int32_t* n_kept, int64_t ntot) {
    const int64_t nk = *n_kept;
    return nk < 0 ? 0 : (nk > ntot ? ntot : nk);
}

__global__ void __launch_bounds__(kRowsThreads) gather_rows_kernel(const RowsArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t nk = clamp_kept(a.n_kept, a.ntot);
    const int lane = threadIdx.x & 31;
    const int vpd = a.d / 8;     // 16-byte vectors per head
    const int vpr = a.hk * vpd;  // per row
    const int64_t rows = nk * a.ly;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRowsWarps;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kRowsWarps + (threadIdx.x >> 5); w < rows;
         w += nwarps) {
        const int64_t layer = w / nk, i = w - layer * nk;
        const int64_t t = a.kept_idx[i];
        const bool ok = t >= 0 && t < a.ntot;
        const uint16_t* s = a.src + layer * a.ks_layer + (ok ? t : 0) * a.ks_token;
        uint4* o = reinterpret_cast<uint4*>(a.dst + (layer * a.dst_rows + i) * a.hk * a.d);
        for (int v0 = 0; v0 < vpr; v0 += 32 * kRowsUnroll) {
            uint4 r[kRowsUnroll];
#pragma unroll
            for (int u = 0; u < kRowsUnroll; ++u) {
                const int v = v0 + u * 32 + lane;
                r[u] = make_uint4(0, 0, 0, 0);
                if (ok && v < vpr) {
                    const int g = v / vpd;
                    r[u] = __ldcs(reinterpret_cast<const uint4*>(s + g * a.ks_head) + (v - g * vpd));
                }
            }
#pragma unroll
            for (int u = 0; u < kRowsUnroll; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < vpr) __stcs(o + v, r[u]);
            }
        }
    }
}

__global__ void __launch_bounds__(kRowsThreads)
    gather_tokens_kernel(const int32_t* ids, const int32_t* kept_idx, const int32_t* n_kept,
                         int32_t* out, int64_t ntot) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t nk = clamp_kept(n_kept, ntot);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kRowsThreads + threadIdx.x; i < nk;
         i += static_cast<int64_t>(gridDim.x) * kRowsThreads) {
        const int64_t t = kept_idx[i];
        out[i] = (t >= 0 && t < ntot) ? ids[t] : -1;
    }
}

// Sliding-window merge ("SpecPrefill — Implementation Guide", v3.1
// §Sliding Window Loop): window w starts at w * stride; every window but the
// last contributes its first `stride` scores and the last window (the first
// whose end w * stride + window reaches n) all of its own, so token t takes
// the score of window min(t / stride, last) at offset t - w * stride. The
// windows' vectors are packed back to back and every window before the last
// has `window` tokens.
__global__ void __launch_bounds__(kRowsThreads)
    merge_windows_kernel(const float* imp_windows, float* out, int64_t n, int64_t window,
                         int64_t stride) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t last = n > window ? (n - window + stride - 1) / stride : 0;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kRowsThreads + threadIdx.x; t < n;
         t += static_cast<int64_t>(gridDim.x) * kRowsThreads) {
        const int64_t w = min(t / stride, last);
        out[t] = imp_windows[w * window + (t - w * stride)];
    }
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

}  // namespace

cudaError_t launch_gather_rows(const sp_shape* s, const int32_t* kept_idx, const int32_t* n_kept,
                               const uint16_t* src, uint16_t* dst, int64_t dst_rows,
                               cudaStream_t st) {
    RowsArgs a;
    a.kept_idx = kept_idx;
    a.n_kept = n_kept;
    a.src = src;
    a.dst = dst;
    a.ntot = s->n_tokens_total;
    a.dst_rows = dst_rows;
    a.ly = s->n_layers;
    a.hk = s->n_kv_heads;
    a.d = s->head_dim;
    a.ks_layer = s->k_stride_layer;
    a.ks_token = s->k_stride_token;
    a.ks_head = s->k_stride_head;
    return launch_k(gather_rows_kernel, static_cast<unsigned>(kRowsCtasPerSm * sm_count()),
                    kRowsThreads, 0, st, a);
}

cudaError_t launch_merge_windows(int64_t n, int window, int stride, const float* imp_windows,
                                 float* out, cudaStream_t st) {
    int64_t blocks = (n + kRowsThreads - 1) / kRowsThreads;
    const int64_t cap = static_cast<int64_t>(kRowsCtasPerSm) * sm_count();
    if (blocks > cap) blocks = cap;
    return launch_k(merge_windows_kernel, static_cast<unsigned>(blocks), kRowsThreads, 0, st,
                    imp_windows, out, n, static_cast<int64_t>(window), static_cast<int64_t>(stride));
}

cudaError_t launch_gather_tokens(const int32_t* ids, const int32_t* kept_idx, const int32_t* n_kept,
                                 int32_t* out, int64_t ntot, cudaStream_t st) {
    int64_t blocks = (ntot + kRowsThreads - 1) / kRowsThreads;
    const int64_t cap = static_cast<int64_t>(kRowsCtasPerSm) * sm_count();
    if (blocks > cap) blocks = cap;
    return launch_k(gather_tokens_kernel, static_cast<unsigned>(blocks), kRowsThreads, 0, st, ids,
                    kept_idx, n_kept, out, ntot);
}

}  // namespace sp

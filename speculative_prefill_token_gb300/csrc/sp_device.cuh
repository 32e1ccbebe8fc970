// Device helpers shared by the logits kernels: per-warp softmax partials.
#pragma once

#include <cmath>
#include <cstdint>

namespace sp {

// Butterfly reduction of 32 rows held by every lane (v[r] = row r of this
// lane's token): afterwards v[0] of lane r holds op over the 32 lanes of
// row r. 31 shuffles instead of 32 separate 5-step reductions.
template <bool kMax>
__device__ __forceinline__ float warp_rows_reduce(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? v[i] : v[i + h];
            const float keep = upper ? v[i + h] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, h);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
    return v[0];
}

// Per-warp softmax partials of 32 rows over the warp's 32 tokens:
// returns (max, sum exp2(x - max)) of row `lane` (invalid tokens carry -inf).
__device__ __forceinline__ float2 warp_row_partials(const float (&x)[32]) {
    float w[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) w[r] = x[r];
    const float m_own = warp_rows_reduce<true>(w);
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const float m = __shfl_sync(0xffffffffu, m_own, r);
        w[r] = (x[r] == -INFINITY) ? 0.0f : exp2f(x[r] - m);
    }
    const float z_own = warp_rows_reduce<false>(w);
    return make_float2(m_own, z_own);
}

__device__ __forceinline__ float2 merge_partial(float2 a, float2 b) {
    if (a.y == 0.0f) return b;
    if (b.y == 0.0f) return a;
    const float m = fmaxf(a.x, b.x);
    return make_float2(m, a.y * exp2f(a.x - m) + b.y * exp2f(b.x - m));
}


__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Largest b in [0, B) with base[b] <= x (base non-decreasing, base[0] = 0).
__device__ __forceinline__ int search_base(const int32_t* base, int B, int64_t x) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (base[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace sp

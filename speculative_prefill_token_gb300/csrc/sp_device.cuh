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


// Running softmax statistics of up to 32*NH rows, held per thread (one
// token per tile): m = running reference (log2 units), z = sum of
// exp2(x - m). The reference moves only when a value exceeds it by more
// than 16, so the common update is one exp2 and one add.
template <int NH>
struct RowStats {
    float m[NH][32];
    float z[NH][32];
};

template <int NH>
__device__ __forceinline__ void stats_reset(RowStats<NH>& st) {
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            st.m[h][r] = -INFINITY;
            st.z[h][r] = 0.0f;
        }
}

// x = raw dot products of this thread's token; scaled value = x * scale2.
template <int NH>
__device__ __forceinline__ void stats_add(RowStats<NH>& st, const float (&x)[NH][32], float scale2) {
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const float y = fmaf(x[h][r], scale2, -st.m[h][r]);
            const bool big = y > 16.0f;
            const float e = exp2f(big ? -y : y);
            st.z[h][r] = big ? fmaf(st.z[h][r], e, 1.0f) : st.z[h][r] + e;
            st.m[h][r] = big ? x[h][r] * scale2 : st.m[h][r];
        }
}

// Reduce the running statistics of one 128-thread warpgroup (4 warps,
// warp `qw` of it) to one (max, sum) pair per row and write rows < R to
// out[r]; sm is a [4][64] float2 scratch, bar_id a named barrier of the
// warpgroup. Resets the statistics.
template <int NH>
__device__ __forceinline__ void stats_flush(RowStats<NH>& st, float2* sm, int qw, int bar_id,
                                            float2* out, int R) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 0; h < NH; ++h) {
        float w[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) w[r] = st.m[h][r];
        const float mw = warp_rows_reduce<true>(w);
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const float M = __shfl_sync(0xffffffffu, mw, r);
            w[r] = st.z[h][r] > 0.0f ? st.z[h][r] * exp2f(st.m[h][r] - M) : 0.0f;
        }
        const float zw = warp_rows_reduce<false>(w);
        sm[qw * 64 + h * 32 + lane] = make_float2(mw, zw);
    }
    asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
    if (qw == 0) {
        for (int r = lane; r < R; r += 32) {
            float2 acc = sm[r];
            acc = merge_partial(acc, sm[64 + r]);
            acc = merge_partial(acc, sm[128 + r]);
            acc = merge_partial(acc, sm[192 + r]);
            out[r] = acc;
        }
    }
    asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
    stats_reset(st);
}

// Work split of the logits kernels: CTA c of C owns flattened items
// [floor(W*c/C), floor(W*(c+1)/C)). owner(w) = the CTA owning item w.
__device__ __forceinline__ int64_t split_start(int64_t W, int64_t C, int64_t c) { return (W * c) / C; }

__device__ __forceinline__ int64_t split_owner(int64_t W, int64_t C, int64_t w) {
    int64_t lo = 0, hi = C - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (split_start(W, C, mid) <= w) lo = mid; else hi = mid - 1;
    }
    return lo;
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

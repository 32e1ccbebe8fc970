// Device helpers shared by the logits kernels: per-warp softmax partials.
#pragma once

#include <cmath>
#include <cstdint>

namespace sp {

// Programmatic dependent launch. grid_dep_wait() returns once the kernel
// that precedes this one in the stream has completed and its memory writes
// are visible (that kernel itself waited for its predecessor, so everything
// earlier in the stream is complete too); without the launch attribute it
// returns at once. grid_dep_launch() lets the next kernel of the stream be
// scheduled: its CTAs may become resident early and then block in their own
// grid_dep_wait(). Every kernel of this library calls grid_dep_wait() before
// its first global-memory access. In the fused call only the prep kernel
// releases its successor at once (the logits kernel then sets up its TMEM,
// barriers and tensor maps under the prep kernel's tail); the logits,
// importance, pool, rank and gather kernels do not (measured faster: an
// early-released successor parks its CTAs on the SMs that free up first).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Logits scratch format. A scaled logit y = s * scale * log2(e) is stored
// as the unsigned 16-bit fixed-point value of M - y, where M is the row's
// maximum over the valid tokens of the warp quarter (32 tokens) of its tile,
// with kLogitQuant steps per unit and clamped at kLogitQuantMax (M - y > 32).
// M never exceeds the row's log2 softmax normaliser, so every probability
// above 2^-32 has M - y < 32 and is reconstructed to within half a step
// (2^-12 in log2 units: a relative error below 1.7e-4).
constexpr float kLogitQuant = 2048.0f;
constexpr float kLogitQuantInv = 1.0f / 2048.0f;
constexpr uint32_t kLogitQuantMax = 65535u;

// Rounds to nearest (ties to even) on the floating-point adder: for
// 0 <= c <= 65535, c + 1.5 * 2^23 has a unit in the last place of 1, so its
// low mantissa bits are the rounded integer. Negative differences give 0,
// NaN and differences from kLogitQuantMax up give kLogitQuantMax.
__device__ __forceinline__ uint32_t quant_logit(float M, float y) {
    const float d = (M - y) * kLogitQuant;  // >= 0 for the tokens that are read back
    const float c = d < static_cast<float>(kLogitQuantMax) ? fmaxf(d, 0.0f) : static_cast<float>(kLogitQuantMax);
    return __float_as_uint(c + 12582912.0f) - 0x4B400000u;
}

// The 16-bit code of a non-negative distance d = 2^11 (M - y) computed by
// the caller: round to nearest on the adder, NaN and d >= kLogitQuantMax
// give kLogitQuantMax (a negative d gives unspecified low bits).
__device__ __forceinline__ uint32_t quant_distance(float d) {
    const float c = fminf(d, static_cast<float>(kLogitQuantMax));
    return __float_as_uint(c + 12582912.0f) - 0x4B400000u;
}

// 2^x by the PTX approximation instruction, results below 2^-126 flushed
// to zero (the softmax partial sums it feeds are at least 1).
__device__ __forceinline__ float exp2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

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

// Reduce per-lane running row statistics of one 128-thread warpgroup (4
// warps, warp qw; lane r holds the (max, sum of exp2(y - max)) pair of row
// hh * 32 + r over its warp's tokens) to one pair per row, write rows < R to
// out[r] and reset the pairs. sm is a [4][64] float2 scratch, bar_id a named
// barrier of the warpgroup.
template <int NH>
__device__ __forceinline__ void flush_rows(float2 (&run)[NH], float2* sm, int qw, int bar_id, float2* out,
                                           int R) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) sm[qw * 64 + hh * 32 + lane] = run[hh];
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
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) run[hh] = make_float2(-INFINITY, 0.0f);
}

// Work split of the logits kernels: CTA c of C owns flattened items
// [start(c), start(c + 1)), q = W / C items each and one more for the first
// r = W mod C CTAs (start(c) = c q + min(c, r)). The last CTA index is the
// one most often placed late (on the SM that still runs the previous
// kernel), so it never carries an extra item. owner(w) = the CTA owning
// item w.
__device__ __forceinline__ int64_t split_start(int64_t W, int64_t C, int64_t c) {
    const int64_t q = W / C, r = W - q * C;
    return c * q + (c < r ? c : r);
}

__device__ __forceinline__ int64_t split_owner(int64_t W, int64_t C, int64_t w) {
    const int64_t q = W / C, r = W - q * C, big = r * (q + 1);
    return w < big ? w / (q + 1) : r + (w - big) / q;
}

// GPU-scope acquire-release atomic add; returns the previous value.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Called by all 128 threads of a warpgroup right after it wrote `contrib`
// softmax records of segment `seg` and passed a warpgroup barrier. The
// warpgroup whose contribution completes the segment's count (2 records per
// CTA that owns items of the segment) merges all of the segment's records
// into lse2[seg][r] = max + log2(sum) and resets the counter. Nothing waits:
// the last one to arrive does the work (acquire-release atomic counter).
__device__ __forceinline__ void segment_done(const int32_t* tile_base, int B, int nslab, int64_t C,
                                             int64_t seg, int contrib, const float2* rec,
                                             unsigned* seg_cnt, float* lse2, int R, int Rs,
                                             float2* sm, volatile int* flag, int qw, int bar_id) {
    const int lane = threadIdx.x & 31;
    const int slab = static_cast<int>(seg / B), b = static_cast<int>(seg - static_cast<int64_t>(slab) * B);
    const int64_t T = tile_base[B];
    const int64_t W = T * nslab;
    const int64_t i0 = static_cast<int64_t>(slab) * T + tile_base[b];
    const int64_t i1 = static_cast<int64_t>(slab) * T + tile_base[b + 1];
    const int64_t c0 = split_owner(W, C, i0), c1 = split_owner(W, C, i1 - 1);
    // CTAs in [c0, c1] that own at least one item: all of them when C <= W
    // (every CTA then owns one or more items), otherwise one per item
    const int64_t owners = C > W ? (i1 - i0) : (c1 - c0 + 1);
    if (qw == 0 && lane == 0) {
        const unsigned target = static_cast<unsigned>(2 * owners);
        // acquire-release: publishes this warpgroup's records (the barrier
        // above ordered its lanes' stores before this add) and, for the last
        // contributor, makes every other contributor's records visible; no
        // separate fence on either side (2B workload 62.2 -> 61.6 us per
        // call, long 240.8 -> 239.1)
        const unsigned prev = atom_add_acq_rel(seg_cnt + seg, static_cast<unsigned>(contrib));
        const int last = (prev + contrib == target) ? 1 : 0;
        if (last) seg_cnt[seg] = 0u;
        *flag = last;
    }
    asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
    const bool last = *flag != 0;
    if (last) {
        // warp qw merges the records of CTAs c0 + qw, c0 + qw + 4, ... that own
        // items; four CTAs' records are loaded before they are merged
        for (int h = 0; h * 32 < R; ++h) {
            const int r = h * 32 + lane;
            float2 acc = make_float2(-INFINITY, 0.0f);
            if (r < R) {
                for (int64_t cb = c0 + qw; cb <= c1; cb += 16) {
                    float2 v[8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int64_t c = cb + 4 * u;
                        const bool own = c <= c1 && (C <= W || split_start(W, C, c + 1) != split_start(W, C, c));
                        v[2 * u] = own ? __ldcg(rec + ((c + seg) * 2 + 0) * Rs + r) : make_float2(-INFINITY, 0.0f);
                        v[2 * u + 1] = own ? __ldcg(rec + ((c + seg) * 2 + 1) * Rs + r) : make_float2(-INFINITY, 0.0f);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc = merge_partial(acc, v[u]);
                }
            }
            sm[qw * 64 + r] = acc;
        }
    }
    asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
    if (last && qw == 0) {
        for (int r = lane; r < R; r += 32) {
            float2 acc = sm[r];
            acc = merge_partial(acc, sm[64 + r]);
            acc = merge_partial(acc, sm[128 + r]);
            acc = merge_partial(acc, sm[192 + r]);
            lse2[seg * Rs + r] = acc.y > 0.0f ? acc.x + log2f(acc.y) : INFINITY;
        }
    }
    asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
}

// Chunk score = mean over the chunk of boost(t) * normalise(x(t)). The
// min-max normalisation is affine, so with S_bx = sum boost*x and
// S_b = sum boost (warp_chunk_sums) the mean is
// (S_bx - min * S_b) / (max - min) / count; a constant prompt (max == min)
// normalises to all ones, giving S_b / count. Clamped at zero (rounding of
// the difference of two nearly equal sums).
__device__ __forceinline__ float chunk_score_from_sums(float sbx, float sb, float mn, float mx,
                                                       int normalize, int64_t count) {
    const float cnt = static_cast<float>(count);
    if (!normalize) return sbx / cnt;
    if (mx == mn) return sb / cnt;
    return fmaxf(fmaf(-mn, sb, sbx), 0.0f) / (mx - mn) / cnt;
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

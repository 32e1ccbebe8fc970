// Chunk selection of one prompt by one CTA: radix select on the order
// (score descending, chunk index ascending) — "SpecPrefill — Implementation
// Guide" §Chunk Selection (top fraction by average score) and v3 §v3
// Improvements item 1 (cumulative attention mass).
//
// Fixed mode keeps the first k = max(1, ceil(nc * p)) positions of that
// order; mass mode keeps the shortest prefix whose running score sum reaches
// mass * (sum of all scores), the crossing chunk included (all chunks when
// the total is zero). Only the set is needed, so instead of sorting, four
// MSB-first 8-bit histogram passes find the key of the last kept position;
// chunks with a smaller key are kept, and ties with that key are resolved by
// chunk index. Mass mode accumulates scores as exact fixed-point integers
// (each fp32 score scaled by a power of two chosen per prompt so that the
// total stays below 2^53, converted with integer operations only), so the
// sums are exact and independent of the order of the atomic additions.
#pragma once

#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {

constexpr int kSelectThreads = 256;
constexpr int kSelectWarps = kSelectThreads / 32;

// Ascending order key of a descending score.
__device__ __forceinline__ uint32_t score_desc_key(float f) {
    const uint32_t u = __float_as_uint(f);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~ord;
}

// round(f * 2^S) for a non-negative finite fp32 f, integer operations only
// (half rounds up); S chosen by the caller so the result stays below 2^53.
__device__ __forceinline__ uint64_t fixed_point(float f, int S) {
    const uint32_t u = __float_as_uint(f) & 0x7fffffffu;
    int e = static_cast<int>(u >> 23);
    uint64_t m = u & 0x7fffffu;
    if (e == 0) e = 1; else m |= 0x800000u;
    const int sh = e - 150 + S;   // value = m * 2^(e - 150)
    if (m == 0) return 0;
    if (sh >= 0) return m << sh;
    if (sh <= -64) return 0;
    return (m + (uint64_t(1) << (-sh - 1))) >> (-sh);
}

// Fixed mode: k = max(1, ceil(nc * p)), at most nc (float64, as the
// oracle's definition; one thread).
__device__ __forceinline__ uint64_t fixed_keep_count(int64_t nc, float keep_p) {
    const double kk = ceil(static_cast<double>(nc) * static_cast<double>(keep_p));
    const int64_t k = kk < 1.0 ? 1 : static_cast<int64_t>(kk);
    return static_cast<uint64_t>(k > nc ? nc : k);
}

// Listing rule ("SpecPrefill — Implementation Guide", v2 listing
// `select_chunks`): k = max(1, ceil(nc * p)) where the product of the chunk
// count and the float32 p is itself a float32 (5 * 0.4f is 2, not 3); at
// most nc.
__device__ __forceinline__ uint64_t listing_keep_count(int64_t nc, float keep_p) {
    const float kk = ceilf(__fmul_rn(static_cast<float>(nc), keep_p));
    const int64_t k = kk < 1.0f ? 1 : static_cast<int64_t>(kk);
    return static_cast<uint64_t>(k > nc ? nc : k);
}

// Listing rule: the smallest kept-token count of an n-token prompt,
// min(min_tok, max(4, n / 10)).
__device__ __forceinline__ int64_t listing_eff_min(int64_t n, int min_tok) {
    return min64(static_cast<int64_t>(min_tok), max64(4, n / 10));
}

// Listing rule: is token t of an n-token prompt one of the forced tokens
// {0, 1, 2, 3} and, when n > 4, {n - 2, n - 1}?
__device__ __forceinline__ bool listing_forced(int64_t t, int64_t n) {
    return t < 4 || (n > 4 && t >= n - 2);
}

// Listing rule: forced tokens in [a0, a1) of an n-token prompt.
__device__ __forceinline__ int64_t listing_forced_in(int64_t a0, int64_t a1, int64_t n) {
    const int64_t head = max64(0, min64(a1, min64(4, n)) - a0);
    const int64_t tail = n > 4 ? max64(0, min64(a1, n) - max64(a0, max64(4, n - 2))) : 0;
    return head + tail;
}

// Mass mode: the power-of-two scale S of the fixed-point scores, from the
// prompt's largest score, so that the sum of nc scores stays below 2^52.
__device__ __forceinline__ int mass_scale(int64_t nc, float smax) {
    if (!(smax > 0.0f)) return 0;
    int lg = 0;
    while ((int64_t(1) << lg) < nc + 1) ++lg;
    const int e_max = static_cast<int>((__float_as_uint(smax) >> 23) & 0xff) - 127;  // floor(log2)
    return 52 - (e_max + 1) - lg;
}

// Mass mode: integer threshold ceil(mass * total); for an integer running
// sum, cum >= mass * total <=> cum >= ceil(mass * total).
__device__ __forceinline__ uint64_t mass_threshold(uint64_t total, float mass) {
    return static_cast<uint64_t>(ceil(static_cast<double>(mass) * static_cast<double>(total)));
}

struct SelectShared {
    unsigned wcnt_h[kSelectWarps][256];            // per-warp histograms
    unsigned long long wsum_h[kSelectWarps][256];
    unsigned cnt[256];
    unsigned long long sum[256];
    unsigned long long wtot[32];
    unsigned wcnt[32];
    float wmax[32];
    int digit;
    unsigned long long need_b;   // fixed: rank to find; mass: ceil(theta) (integer threshold)
    int all_b;
    unsigned cnt_before;
    unsigned long long sum_before;
    int found;
    unsigned long long total;
    float smax;
};

// flags[c] |= 1 for every kept chunk c < nc (flags zeroed by the caller).
// scores: the prompt's nc chunk scores in shared memory. All kSelectThreads
// threads of the CTA call this; thread t owns chunks [t*E, t*E + E).
__device__ __forceinline__ void radix_select(const float* scores, int64_t nc, int mode, float keep_p,
                                             float mass, uint8_t* flags, SelectShared& sm) {
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int E = static_cast<int>((nc + kSelectThreads - 1) / kSelectThreads);
    const int64_t c_lo = static_cast<int64_t>(t) * E;
    const int64_t c_hi = c_lo + E < nc ? c_lo + E : nc;
    const bool is_mass = mode == SP_MODE_MASS;
    // GB300 runs FP64 at a small fraction of the FP32 rate: the few float64
    // operations (k = ceil(nc * p), theta = mass * total) run in one thread
    // and every comparison afterwards is an integer one (for an integer
    // running sum, cum >= theta <=> cum >= ceil(theta)).
    int S = 0;
    if (is_mass) {
        float mx = 0.0f;
        for (int64_t c = c_lo; c < c_hi; ++c) mx = fmaxf(mx, scores[c]);
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) sm.wmax[warp] = mx;
        __syncthreads();
        if (t == 0) {
            float m = 0.0f;
            for (int w = 0; w < kSelectWarps; ++w) m = fmaxf(m, sm.wmax[w]);
            sm.smax = m;
        }
        __syncthreads();
        S = mass_scale(nc, sm.smax);
        uint64_t part = 0;
        for (int64_t c = c_lo; c < c_hi; ++c) part += fixed_point(scores[c], S);
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) sm.wtot[warp] = part;
        __syncthreads();
        if (t == 0) {
            unsigned long long tot = 0;
            for (int w = 0; w < kSelectWarps; ++w) tot += sm.wtot[w];
            sm.all_b = tot == 0 ? 1 : 0;
            sm.need_b = mass_threshold(tot, mass);
        }
    } else if (t == 0) {
        sm.need_b = fixed_keep_count(nc, keep_p);
        sm.all_b = 0;
    }
    __syncthreads();
    uint64_t need = sm.need_b;     // fixed: rank; mass: integer threshold
    bool all = sm.all_b != 0;
    uint32_t prefix = 0, pmask = 0;
    uint64_t base_sum = 0;  // mass: fixed-point sum of all keys below the current bucket
    unsigned final_ties = 0;
    for (int pass = 0; pass < 4 && !all; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = t; i < kSelectWarps * 256; i += kSelectThreads) {
            (&sm.wcnt_h[0][0])[i] = 0u;
            if (is_mass) (&sm.wsum_h[0][0])[i] = 0ull;
        }
        __syncthreads();
        // each warp counts into its own histogram: no contention across warps
        for (int64_t c = c_lo; c < c_hi; ++c) {
            const float sc = scores[c];
            const uint32_t key = score_desc_key(sc);
            if ((key & pmask) == prefix) {
                const int d = static_cast<int>((key >> shift) & 0xffu);
                atomicAdd(&sm.wcnt_h[warp][d], 1u);
                if (is_mass) atomicAdd(&sm.wsum_h[warp][d], static_cast<unsigned long long>(fixed_point(sc, S)));
            }
        }
        __syncthreads();
        {
            const int d = t;  // kSelectThreads == 256 bins
            unsigned c = 0;
            unsigned long long sv = 0;
#pragma unroll
            for (int w = 0; w < kSelectWarps; ++w) {
                c += sm.wcnt_h[w][d];
                if (is_mass) sv += sm.wsum_h[w][d];
            }
            sm.cnt[d] = c;
            sm.sum[d] = sv;
        }
        __syncthreads();
        if (warp == 0) {
            unsigned lc = 0;
            unsigned long long ls = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lc += sm.cnt[8 * lane + i];
                ls += sm.sum[8 * lane + i];
            }
            unsigned ic = lc;
            unsigned long long is = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned uc = __shfl_up_sync(0xffffffffu, ic, o);
                const unsigned long long us = __shfl_up_sync(0xffffffffu, is, o);
                if (lane >= o) {
                    ic += uc;
                    is += us;
                }
            }
            unsigned cb = ic - lc;             // counts of this pass's bins before the lane
            unsigned long long sb = is - ls;
            int hit = -1;
            unsigned hit_cb = 0;
            unsigned long long hit_sb = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = 8 * lane + i;
                const unsigned c = sm.cnt[d];
                const unsigned long long sv = sm.sum[d];
                bool reach;
                if (is_mass) reach = c > 0 && base_sum + sb + sv >= need;
                else reach = static_cast<uint64_t>(cb) + c >= need;
                if (hit < 0 && reach) {
                    hit = d;
                    hit_cb = cb;
                    hit_sb = sb;
                }
                cb += c;
                sb += sv;
            }
            const unsigned ballot = __ballot_sync(0xffffffffu, hit >= 0);
            if (ballot == 0) {
                if (lane == 0) sm.found = 0;
            } else if (lane == __ffs(ballot) - 1) {
                sm.found = 1;
                sm.digit = hit;
                sm.cnt_before = hit_cb;
                sm.sum_before = hit_sb;
            }
        }
        __syncthreads();
        if (!sm.found) {
            all = true;  // the running sum never reaches theta: every chunk is kept
        } else {
            const int d = sm.digit;
            prefix |= static_cast<uint32_t>(d) << shift;
            pmask |= 0xffu << shift;
            if (is_mass) base_sum += sm.sum_before;
            else need -= sm.cnt_before;
            final_ties = sm.cnt[d];
        }
        __syncthreads();
    }

    if (all) {
        for (int64_t c = c_lo; c < c_hi; ++c) flags[c] |= 1;
        return;
    }
    // keys below the final key are kept; ties with it in chunk-index order
    unsigned my_ties = 0;
    unsigned long long my_tie_sum = 0;
    for (int64_t c = c_lo; c < c_hi; ++c)
        if (score_desc_key(scores[c]) == prefix) {
            ++my_ties;
            if (is_mass) my_tie_sum += fixed_point(scores[c], S);
        }
    unsigned tie_before = 0;
    unsigned long long tie_sum_before = 0;
    if (final_ties > 1) {
        // exclusive scans of the tie counts (and sums) in chunk order
        unsigned ic = my_ties;
        unsigned long long is = my_tie_sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned uc = __shfl_up_sync(0xffffffffu, ic, o);
            const unsigned long long us = __shfl_up_sync(0xffffffffu, is, o);
            if (lane >= o) {
                ic += uc;
                is += us;
            }
        }
        if (lane == 31) {
            sm.wcnt[warp] = ic;
            sm.wtot[warp] = is;
        }
        __syncthreads();
        if (warp == 0) {
            unsigned wc = lane < kSelectWarps ? sm.wcnt[lane] : 0u;
            unsigned long long wsum = lane < kSelectWarps ? sm.wtot[lane] : 0ull;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned uc = __shfl_up_sync(0xffffffffu, wc, o);
                const unsigned long long us = __shfl_up_sync(0xffffffffu, wsum, o);
                if (lane >= o) {
                    wc += uc;
                    wsum += us;
                }
            }
            sm.wcnt[lane] = wc;
            sm.wtot[lane] = wsum;
        }
        __syncthreads();
        tie_before = ic - my_ties + (warp > 0 ? sm.wcnt[warp - 1] : 0u);
        tie_sum_before = is - my_tie_sum + (warp > 0 ? sm.wtot[warp - 1] : 0ull);
        __syncthreads();
    }
    for (int64_t c = c_lo; c < c_hi; ++c) {
        const uint32_t key = score_desc_key(scores[c]);
        bool keep = key < prefix;
        if (key == prefix) {
            if (is_mass) keep = base_sum + tie_sum_before < need;
            else keep = tie_before < need;
            ++tie_before;
            if (is_mass) tie_sum_before += fixed_point(scores[c], S);
        }
        if (keep) flags[c] |= 1;
    }
}

}  // namespace sp

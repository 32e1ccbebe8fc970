// Per-item phases of the SpecPrefill scoring path after the token
// importance, written as device functions for a group of threads (the
// kernels run one item per CTA):
//
//   pool_tile     one 128-token tile: W-window mean of the importance
//                 (llama.cpp PR "Speculative prefill" §Approach item 3), the
//                 tile's min / max and the per-chunk sums of boost * x and of
//                 boost ("SpecPrefill — Implementation Guide" v3 item 2,
//                 §Chunk Selection)
//   rank_slice    chunk scores (min-max normalisation, guide v3.1 item 5)
//                 and the selection of one slice of 32 chunks (guide
//                 §Chunk Selection, v3 item 1; PR §Approach item 4)
//   gather_slice  kept token indices and positions of one slice (guide
//                 §How It Works / Sparse Prefill) and the per-prompt offsets
//
// Values written by other CTAs or kernels are read through L2
// (ld.global.cg), never from a possibly stale L1 line.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_select.cuh"

namespace sp {

// Named barrier over the first-to-last `n` threads of a warp-aligned group.
struct GroupBar {
    int id, n;
    __device__ __forceinline__ void sync() const {
        asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
    }
};

// --------------------------------------------------------------- locate
// Item x (a tile or slice) of a per-prompt base table (base[0] = 0,
// non-decreasing, base[B] = the item count): its prompt b = the last b < B
// with base[b] <= x, base[b], base[B], the first prompt f <= b with
// base[f] = base[b] (prompts f .. b-1 are empty), and aux[k][b],
// aux[k][b + 1] for NA more tables of B + 1 entries. For B < 32 kLocRegs
// every lane of the warp loads entries lane + 32 j of each table, so all of
// it takes one round of loads, and b and f come from ballots; larger
// batches search. Called by whole warps with x uniform across the warp.
constexpr int kLocRegs = 2;

template <int NA>
struct Located {
    int b, first;
    int32_t base_b, total;
    int32_t lo[NA > 0 ? NA : 1], hi[NA > 0 ? NA : 1];
};

__device__ __forceinline__ int32_t lane_pick(const int32_t (&v)[kLocRegs], int j) {
    int32_t out = 0;
#pragma unroll
    for (int k = 0; k < kLocRegs; ++k) {
        const int32_t u = __shfl_sync(0xffffffffu, v[k], j & 31);
        if ((j >> 5) == k) out = u;
    }
    return out;
}

template <int NA>
__device__ __forceinline__ Located<NA> locate(const int32_t* base, const int32_t* const (&aux)[NA > 0 ? NA : 1],
                                              int B, int64_t x) {
    Located<NA> r;
    if (B < 32 * kLocRegs) {
        const int lane = threadIdx.x & 31;
        int32_t v[kLocRegs], w[NA > 0 ? NA : 1][kLocRegs];
#pragma unroll
        for (int k = 0; k < kLocRegs; ++k) {
            const int j = lane + 32 * k;
            v[k] = j <= B ? base[j] : 0;
#pragma unroll
            for (int q = 0; q < NA; ++q) w[q][k] = j <= B ? aux[q][j] : 0;
        }
        int cnt = 0;
#pragma unroll
        for (int k = 0; k < kLocRegs; ++k)
            cnt += __popc(__ballot_sync(0xffffffffu, lane + 32 * k < B && v[k] <= x));
        r.b = cnt > 0 ? cnt - 1 : 0;
        r.base_b = lane_pick(v, r.b);
        r.total = lane_pick(v, B);
        int before = 0;
#pragma unroll
        for (int k = 0; k < kLocRegs; ++k)
            before += __popc(__ballot_sync(0xffffffffu, lane + 32 * k < B && v[k] < r.base_b));
        r.first = before;
#pragma unroll
        for (int q = 0; q < NA; ++q) {
            r.lo[q] = lane_pick(w[q], r.b);
            r.hi[q] = lane_pick(w[q], r.b + 1);
        }
    } else {
        r.total = base[B];
        r.b = search_base(base, B, x);
        r.base_b = base[r.b];
        int f = r.b;
        while (f > 0 && base[f - 1] == r.base_b) --f;
        r.first = f;
#pragma unroll
        for (int q = 0; q < NA; ++q) {
            r.lo[q] = aux[q][r.b];
            r.hi[q] = aux[q][r.b + 1];
        }
    }
    return r;
}

// A single prompt (B = 1) has seq_off = {0, Ntot} once the prep kernel has
// accepted the input (it raises the bad-input flag otherwise), so every
// per-prompt table follows from Ntot without loads: `items` is base[1] (the
// tile or slice count) and aux[q] = {0, hi[q]}.
template <int NA>
__device__ __forceinline__ Located<NA> one_prompt(int32_t items, const int64_t (&hi)[NA > 0 ? NA : 1]) {
    Located<NA> r;
    r.b = 0;
    r.first = 0;
    r.base_b = 0;
    r.total = items;
#pragma unroll
    for (int q = 0; q < NA; ++q) {
        r.lo[q] = 0;
        r.hi[q] = static_cast<int32_t>(hi[q]);
    }
    return r;
}

// Sums over the chunk's tokens [a0, a1) (prompt positions; the pooled
// score of token t at xs[t - x0]) of boost(t) * x(t) and of boost(t), by
// one warp in a fixed order: lane k adds tokens a0 + k, a0 + k + 32, ...
// in turn, then lane k + o is added into lane k for o = 1, 2, 4, 8, 16.
// The sums are in lane 0. boost(t) = bf_mult for t < bf_n, times bl_mult
// for t >= n - bl_n.
__device__ __forceinline__ float2 warp_chunk_sums(const float* xs, int64_t x0, int64_t a0, int64_t a1,
                                                  int64_t n, int bf_n, float bf_mult, int bl_n,
                                                  float bl_mult, int lane) {
    float sbx = 0.0f, sb = 0.0f;
    for (int64_t t = a0 + lane; t < a1; t += 32) {
        float bx = xs[t - x0], bb = 1.0f;
        if (t < bf_n) {
            bx *= bf_mult;
            bb *= bf_mult;
        }
        if (t >= n - bl_n) {
            bx *= bl_mult;
            bb *= bl_mult;
        }
        sbx += bx;
        sb += bb;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float ux = __shfl_down_sync(0xffffffffu, sbx, o);
        const float ub = __shfl_down_sync(0xffffffffu, sb, o);
        if (lane + o < 32) {
            sbx += ux;
            sb += ub;
        }
    }
    return make_float2(sbx, sb);
}

// ------------------------------------------------------------------ pool
constexpr int kPoolThreads = 128;
constexpr int kPoolMaxHalo = 64;

struct PoolArgs {
    const float* imp;
    float* tok;
    float2* rpart;   // per tile (min, max) of the pooled scores
    float2* csum;    // per chunk (sum boost * x, sum boost)
    const int32_t* seq_off;
    const int32_t* tile_base;
    const int32_t* chunk_off;
    int64_t Ntot;
    int B, W, C, bf_n, bl_n;
    float bf_mult, bl_mult;
};

struct PoolShared {
    float win[kTileTokens + 2 * kPoolMaxHalo];
    float xs[kTileTokens];
    float red_mn[kPoolThreads / 32], red_mx[kPoolThreads / 32];
};

// One tile by kPoolThreads threads (tid = thread index within the group),
// located by loc (tile_base; aux seq_off, chunk_off). Chunks never straddle
// tiles (C divides 128); the halo is W/2 <= 64 tokens clipped to the
// prompt. Per-chunk sums: warp_chunk_sums. With bad1 (single prompt, see
// one_prompt) the window is requested before the flag is read.
__device__ __forceinline__ void pool_tile(const PoolArgs& a, int64_t tile, int tid, GroupBar g,
                                          PoolShared& sh, const Located<2>& loc, const int32_t* bad1) {
    const int64_t i = tile - loc.base_b;
    const int64_t start = loc.lo[0];
    const int64_t n = static_cast<int64_t>(loc.hi[0]) - start;
    const int64_t t0 = i * kTileTokens, t1 = min64(n, t0 + kTileTokens);
    const int h = a.W / 2;
    const int64_t lo = max64(0, t0 - h), hi = min64(n, t1 + h);
    constexpr int kWin = (kTileTokens + 2 * kPoolMaxHalo + kPoolThreads - 1) / kPoolThreads;
    float r[kWin];
#pragma unroll
    for (int k = 0; k < kWin; ++k) {
        const int64_t u = lo + tid + k * kPoolThreads;
        r[k] = u < hi ? __ldcg(a.imp + start + u) : 0.0f;
    }
    if (bad1 && *bad1) return;
#pragma unroll
    for (int k = 0; k < kWin; ++k) {
        const int64_t u = lo + tid + k * kPoolThreads;
        if (u < hi) sh.win[u - lo] = r[k];
    }
    g.sync();
    float mn = INFINITY, mx = -INFINITY;
    const int64_t tt = t0 + tid;
    if (tt < t1) {
        const int64_t u0 = max64(0, tt - h), u1 = min64(n - 1, tt + h);
        float s = 0.0f;
        for (int64_t u = u0; u <= u1; ++u) s += sh.win[u - lo];
        const float x = s / static_cast<float>(u1 - u0 + 1);
        a.tok[start + tt] = x;
        sh.xs[tid] = x;
        mn = x;
        mx = x;
    }
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const int warp = tid >> 5, lane = tid & 31;
    if (lane == 0) {
        sh.red_mn[warp] = mn;
        sh.red_mx[warp] = mx;
    }
    g.sync();
    if (tid == 0) {
        for (int w = 1; w < kPoolThreads / 32; ++w) {
            mn = fminf(mn, sh.red_mn[w]);
            mx = fmaxf(mx, sh.red_mx[w]);
        }
        a.rpart[tile] = make_float2(mn, mx);
    }
    // one warp per chunk (the staged chunk kernel sums in the same order)
    const int64_t c_lo = t0 / a.C, c_hi = (t1 + a.C - 1) / a.C;
    for (int64_t c = c_lo + warp; c < c_hi; c += kPoolThreads / 32) {
        const int64_t a0 = c * a.C, a1 = min64(t1, a0 + a.C);
        const float2 r = warp_chunk_sums(sh.xs, t0, a0, a1, n, a.bf_n, a.bf_mult, a.bl_n, a.bl_mult, lane);
        if (lane == 0) a.csum[loc.lo[1] + c] = r;
    }
    g.sync();  // the group's shared memory may be reused for the next tile
}

// ------------------------------------------------------ rank and gather
constexpr int kRankThreads = 256;
constexpr int kRankWarps = kRankThreads / 32;
static_assert(kSliceChunks == 32, "the gather scan uses one lane per chunk of a slice");

struct PostArgs {
    const int32_t* __restrict__ seq_off;
    const int32_t* chunk_off;   // workspace copy
    const int32_t* tile_base;
    const int32_t* slice_base;
    const float2* rpart;        // per pool tile: (min, max) of the pooled scores
    const float2* csum;         // per chunk (sum boost * x, sum boost)
    float* chunk_score;
    uint8_t* keep;
    int32_t* scount;            // kept tokens per slice
    int32_t* kept_idx;
    int32_t* kept_pos;
    int32_t* kept_off;
    int32_t* n_kept;
    int32_t* lcount;            // listing rule: kept tokens per prompt before the fill
    int32_t* ucount;            // listing rule: unselected, unforced tokens per slice
    WsHeader* hdr;
    int B, C, mode, normalize, force_bos, force_last;
    int rule, min_tok, max_keep;
    int rank_split;             // rank CTAs per slice (1 or kRankSplitMax); scount / ucount per part
    int64_t Ntot;
    float keep_p, mass;
};

struct RankShared {
    float red_mn[kRankWarps], red_mx[kRankWarps], red_sm[kRankWarps];
    unsigned long long red_u[kRankWarps], red_acc[kRankWarps];
    int32_t warp_cnt[kRankWarps], warp_spare[kRankWarps];
    int64_t red[kRankWarps];
    int64_t base[kSliceChunks];
    uint8_t keepf[kSliceChunks];
};

__device__ __forceinline__ int64_t chunk_tokens(int64_t n, int C, int64_t c) { return min64(C, n - c * C); }

// Part `piece` (< SPLIT) of slice s (< number of slices) by kRankThreads
// threads: the part's kSliceChunks / SPLIT chunks, each warp ranking one or
// more of them over all or part of the prompt's chunks; cs_s holds room for
// the prompt's chunk scores (kMaxPromptChunks floats at most).
//
// Rebuilds every chunk score of the prompt (the min-max normalisation is
// affine, so the chunk mean comes from the pool kernel's sums) and decides
// the part's chunks by their position in the order (score descending,
// chunk index ascending): fixed mode keeps a chunk when fewer than
// k = max(1, ceil(nc p)) chunks precede it, mass mode when the exact
// fixed-point sum of the scores preceding it is below ceil(mass * total)
// (the shortest prefix that reaches the mass, crossing chunk included).
// The final chunk is forced. Writes the chunk scores, keep flags and the
// part's kept-token count (chunk 0 counts its BOS token when it is not
// selected) at scount[s * SPLIT + piece]. The set equals that of the
// radix selection behind sp_select.
// The slice is located by loc (slice_base; aux seq_off, chunk_off,
// tile_base). With bad1 (single prompt, see one_prompt) the chunk sums and
// tile extrema are requested before the flag is read.
template <int SPLIT>
__device__ __forceinline__ void rank_slice(const PostArgs& a, int64_t s, int piece, int t, GroupBar g,
                                           float* cs_s, RankShared& sh, const Located<3>& loc,
                                           const int32_t* bad1) {
    const int lane = t & 31, warp = t >> 5;
    const int b = loc.b;
    const int64_t n = static_cast<int64_t>(loc.hi[0]) - loc.lo[0];
    const int64_t coff = loc.lo[1];
    const int64_t nc = static_cast<int64_t>(loc.hi[1]) - coff;
    if (nc > kMaxPromptChunks) {
        // reported; the slice keeps nothing so that the gather stays in bounds
        if (t == 0) {
            atomicCAS(&a.hdr->status, 0, static_cast<int>(SP_ERR_DEVICE));
            a.scount[s * SPLIT + piece] = 0;
            a.ucount[s * SPLIT + piece] = 0;
        }
        return;
    }
    constexpr int kPart = kSliceChunks / SPLIT;                             // chunks of the part
    constexpr int kWarpQ = kPart > kRankWarps ? kPart / kRankWarps : 1;     // chunks per warp
    constexpr int kChunkW = kPart < kRankWarps ? kRankWarps / kPart : 1;    // warps per chunk
    constexpr int kLanesQ = kPart / kWarpQ;                                 // warps before a warp's next chunk
    static_assert(kPart * SPLIT == kSliceChunks && kLanesQ * kChunkW == kRankWarps,
                  "a rank CTA's warps split its chunks evenly");
    const int64_t c_lo = (s - loc.base_b) * kSliceChunks + piece * kPart;
    const int64_t c_hi = min64(nc, c_lo + kPart);
    if (c_lo >= c_hi) {  // past the prompt's last chunk: no chunks, no tokens
        if (t == 0) {
            a.scount[s * SPLIT + piece] = 0;
            a.ucount[s * SPLIT + piece] = 0;
        }
        return;
    }

    // each thread's first chunk sums and up to four tile min / max pairs are
    // requested together (one round trip); larger prompts loop (four pairs:
    // long workload 245.2 -> 244.2 us per call)
    constexpr int kPre = 8;
    float2 v[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int64_t c = t + k * kRankThreads;
        v[k] = c < nc ? __ldcg(a.csum + coff + c) : make_float2(0.0f, 0.0f);
    }
    const int64_t p0 = loc.lo[2], p1 = loc.hi[2];
    constexpr int kRp = 4;
    float2 r0[kRp];
#pragma unroll
    for (int k = 0; k < kRp; ++k)
        r0[k] = (a.normalize && p0 + t + k * kRankThreads < p1) ? __ldcg(a.rpart + p0 + t + k * kRankThreads)
                                                               : make_float2(INFINITY, -INFINITY);
    if (bad1 && *bad1) return;
    float mn = 0.0f, mx = 0.0f;
    if (a.normalize) {
        // min and max do not depend on the order (a NaN is dropped either way)
        mn = INFINITY;
        mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < kRp; ++k) {
            mn = fminf(mn, r0[k].x);
            mx = fmaxf(mx, r0[k].y);
        }
        for (int64_t p = p0 + t + kRp * kRankThreads; p < p1; p += kRankThreads) {
            const float2 r = __ldcg(a.rpart + p);
            mn = fminf(mn, r.x);
            mx = fmaxf(mx, r.y);
        }
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        if (lane == 0) {
            sh.red_mn[warp] = mn;
            sh.red_mx[warp] = mx;
        }
        g.sync();
        // every thread combines the warps' values in the same order
        mn = sh.red_mn[0];
        mx = sh.red_mx[0];
        for (int w = 1; w < kRankWarps; ++w) {
            mn = fminf(mn, sh.red_mn[w]);
            mx = fmaxf(mx, sh.red_mx[w]);
        }
    }
    float smax = 0.0f;
    for (int64_t c0 = t;; c0 += kRankThreads * kPre) {
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
            const int64_t c = c0 + k * kRankThreads;
            if (c < nc) {
                const float cs = chunk_score_from_sums(v[k].x, v[k].y, mn, mx, a.normalize,
                                                       chunk_tokens(n, a.C, c));
                cs_s[c] = cs;
                smax = fmaxf(smax, cs);
                if (c >= c_lo && c < c_hi) a.chunk_score[coff + c] = cs;
            }
        }
        if (c0 + kRankThreads * kPre >= nc) break;
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
            const int64_t c = c0 + kRankThreads * kPre + k * kRankThreads;
            v[k] = c < nc ? __ldcg(a.csum + coff + c) : make_float2(0.0f, 0.0f);
        }
    }
    const bool is_mass = a.mode == SP_MODE_MASS;
    const bool listing = a.rule == SP_RULE_LISTING;
    if (is_mass) {
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        if (lane == 0) sh.red_sm[warp] = smax;
    }
    g.sync();  // cs_s complete (and the per-warp maxima)
    // every thread derives the scale, the threshold and the keep-all flag
    // itself from the same shared values
    uint64_t need = 0;
    bool all = false;
    int S = 0;
    if (is_mass) {
        float m = 0.0f;
        for (int w = 0; w < kRankWarps; ++w) m = fmaxf(m, sh.red_sm[w]);
        S = mass_scale(nc, m);
        uint64_t part = 0;
        for (int64_t c = t; c < nc; c += kRankThreads) part += fixed_point(cs_s[c], S);
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) sh.red_u[warp] = part;
        g.sync();
        unsigned long long tot = 0;
        for (int w = 0; w < kRankWarps; ++w) tot += sh.red_u[w];
        all = tot == 0;
        need = mass_threshold(tot, a.mass);
    } else {
        need = listing ? listing_keep_count(nc, a.keep_p) : fixed_keep_count(nc, a.keep_p);
    }
    // the listing keeps every token when p >= 1 (fixed mode) or the prompt
    // is no longer than its smallest kept count
    if (listing && ((!is_mass && a.keep_p >= 1.0f) || n <= listing_eff_min(n, a.min_tok))) all = true;

    // warp w ranks chunks c_lo + w % kLanesQ + kLanesQ * q (q < kWarpQ) of
    // the part over every kChunkW-th group of 32 chunks of the prompt: the
    // count (fixed) or fixed-point mass (mass mode) of the chunks ordered
    // before it; the kChunkW warps of one chunk add their sums. The order
    // key (descending score, ascending index) is one 64-bit integer so that
    // the comparison is branch-free. The listing rule's fixed mode counts
    // only chunks with a strictly larger score (the index half of the key is
    // masked off), so every chunk tied with the k-th score is kept.
    const uint64_t kmask = (listing && !is_mass) ? 0xffffffff00000000ull : ~0ull;
    const int wq = warp % kLanesQ, wp = warp / kLanesQ;
    int64_t ci[kWarpQ];
    uint64_t ki[kWarpQ];
    uint64_t acc[kWarpQ];
#pragma unroll
    for (int q = 0; q < kWarpQ; ++q) {
        ci[q] = c_lo + wq + kLanesQ * q;
        ki[q] = ci[q] < c_hi ? ((static_cast<uint64_t>(score_desc_key(cs_s[ci[q]])) << 32) |
                                static_cast<uint32_t>(ci[q])) & kmask
                             : 0u;
        acc[q] = 0;
    }
    if (!all) {
        // four scores are read before they are compared, so that the shared-
        // memory latency of one overlaps the comparisons of the others (the
        // scan is latency-bound: long workload 7.5 us per CTA with one read in
        // flight)
        constexpr int kStep = 32 * kChunkW;
        const int nci = static_cast<int>(nc);
        int j = lane + 32 * wp;
        for (; j + 3 * kStep < nci; j += 4 * kStep) {
            float sj[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) sj[u] = cs_s[j + kStep * u];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint64_t kj =
                    ((static_cast<uint64_t>(score_desc_key(sj[u])) << 32) | static_cast<uint32_t>(j + kStep * u)) & kmask;
                const uint64_t wj = is_mass ? fixed_point(sj[u], S) : 1u;
#pragma unroll
                for (int q = 0; q < kWarpQ; ++q) acc[q] += kj < ki[q] ? wj : 0u;
            }
        }
        for (; j < nci; j += kStep) {
            const float sj = cs_s[j];
            const uint64_t kj = ((static_cast<uint64_t>(score_desc_key(sj)) << 32) | static_cast<uint32_t>(j)) & kmask;
            const uint64_t wj = is_mass ? fixed_point(sj, S) : 1u;
#pragma unroll
            for (int q = 0; q < kWarpQ; ++q) acc[q] += kj < ki[q] ? wj : 0u;
        }
#pragma unroll
        for (int q = 0; q < kWarpQ; ++q)
            for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
    }
    if (kChunkW > 1) {  // then kWarpQ = 1
        if (lane == 0) sh.red_acc[warp] = acc[0];
        g.sync();
        acc[0] = 0;
        for (int p = 0; p < kChunkW; ++p) acc[0] += sh.red_acc[wq + p * kLanesQ];
    }
    if (lane == 0) {
        int32_t my_cnt = 0, my_spare = 0;
#pragma unroll
        for (int q = 0; q < kWarpQ; ++q) {
            const int64_t c = ci[q];
            if (wp != 0 || c >= c_hi) continue;
            // fixed: fewer than k chunks before it; mass: mass before it below the threshold
            uint8_t f = (all || acc[q] < need) ? 1 : 0;
            if (!listing && a.force_last && c == nc - 1) f |= 2;
            a.keep[coff + c] = f;
            int64_t extra = (c == 0 && a.force_bos && n > 0) ? 1 : 0;  // BOS of an unselected chunk 0
            if (listing) extra = listing_forced_in(c * a.C, c * a.C + chunk_tokens(n, a.C, c), n);
            my_cnt += static_cast<int32_t>(f ? chunk_tokens(n, a.C, c) : extra);
            if (!f) my_spare += static_cast<int32_t>(chunk_tokens(n, a.C, c) - extra);
        }
        sh.warp_cnt[warp] = my_cnt;
        sh.warp_spare[warp] = my_spare;
    }
    g.sync();
    if (t == 0) {
        int32_t tot = 0;
        for (int w = 0; w < kRankWarps; ++w) tot += sh.warp_cnt[w];
        a.scount[s * SPLIT + piece] = tot;
        if (listing) {
            int32_t spare = 0;
            for (int w = 0; w < kRankWarps; ++w) spare += sh.warp_spare[w];
            a.ucount[s * SPLIT + piece] = spare;
            atomicAdd(a.lcount + b, tot);
        }
    }
    g.sync();  // shared memory may be reused for the next slice
}

// Slice s in [0, S] by kRankThreads threads, S = number of slices: offsets
// the slice by the kept tokens of all earlier slices and writes its kept
// token indices and positions; s == S writes the batch total and the
// offsets of prompts without tokens at the end of the batch.
// The slice is located by loc (slice_base, x = s; aux seq_off, chunk_off);
// loc.total is the slice count S. With bad1 (single prompt, see one_prompt)
// the slice's keep flags are requested with the counts, before the flag is
// read.
__device__ __forceinline__ void gather_slice(const PostArgs& a, int64_t s, int t, GroupBar g,
                                             RankShared& sh, const Located<2>& loc, const int32_t* bad1) {
    const int lane = t & 31, warp = t >> 5;
    const int64_t S = loc.total;
    const int b = loc.b;
    const int64_t sb = loc.base_b;
    const int64_t start = loc.lo[0];
    const int64_t n = static_cast<int64_t>(loc.hi[0]) - start;
    const int64_t coff = loc.lo[1];
    const int64_t nc = static_cast<int64_t>(loc.hi[1]) - coff;
    uint8_t f1 = 0;
    if (bad1 && warp == 0 && s < S && (s - sb) * kSliceChunks + lane < nc)
        f1 = __ldcg(a.keep + coff + (s - sb) * kSliceChunks + lane);
    int64_t part = 0;
    for (int64_t i = t; i < s * a.rank_split; i += kRankThreads) part += __ldcg(a.scount + i);
    if (bad1 && *bad1) return;
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) sh.red[warp] = part;
    g.sync();
    int64_t P = 0;
    for (int w = 0; w < kRankWarps; ++w) P += sh.red[w];
    if (s == S) {
        if (t == 0) {
            // prompts without slices at the end of the batch (loc: the last prompt)
            if (sb == S)
                for (int bb = loc.first; bb < a.B; ++bb) a.kept_off[bb] = static_cast<int32_t>(P);
            a.kept_off[a.B] = static_cast<int32_t>(P);
            *a.n_kept = static_cast<int32_t>(P);
        }
        g.sync();
        return;
    }
    if (t == 0 && s == sb) {
        // first slice of prompt b: its offset, and that of empty prompts before it
        for (int bb = loc.first; bb <= b; ++bb) a.kept_off[bb] = static_cast<int32_t>(P);
    }
    const bool ok = nc <= kMaxPromptChunks;  // else reported by the rank; nothing kept
    const int64_t c_lo = (s - sb) * kSliceChunks;
    // exclusive scan of the slice's per-chunk kept tokens (lane = chunk)
    if (warp == 0) {
        const int64_t c = c_lo + lane;
        int64_t cnt = 0;
        uint8_t f = 0;
        if (ok && c < nc) {
            f = bad1 ? f1 : __ldcg(a.keep + coff + c);
            cnt = f ? chunk_tokens(n, a.C, c) : ((c == 0 && a.force_bos && n > 0) ? 1 : 0);
        }
        sh.keepf[lane] = f;
        int64_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        sh.base[lane] = P + incl - cnt;
    }
    g.sync();
    if (ok) {
        for (int q = warp; q < kSliceChunks; q += kRankWarps) {
            const int64_t c = c_lo + q;
            if (c >= nc) break;
            const int64_t base = sh.base[q];
            if (sh.keepf[q]) {
                const int64_t a0 = c * a.C, a1 = min64(n, a0 + a.C);
                for (int64_t tt = a0 + lane; tt < a1; tt += 32) {
                    a.kept_idx[base + (tt - a0)] = static_cast<int32_t>(start + tt);
                    a.kept_pos[base + (tt - a0)] = static_cast<int32_t>(tt);
                }
            } else if (c == 0 && a.force_bos && n > 0 && lane == 0) {
                a.kept_idx[base] = static_cast<int32_t>(start);
                a.kept_pos[base] = 0;
            }
        }
    }
    g.sync();
}

// Host-side argument builders (sp_stages.cu, sp_post.cu).
PoolArgs pool_args(const Plan& pl, const sp_params* p, const int32_t* seq_off, const float* imp,
                   float* tok, void* ws);
PostArgs post_args(const Plan& pl, const sp_params* p, const int32_t* seq_off, float* chunk_score,
                   uint8_t* keep, int32_t* kept_idx, int32_t* kept_pos, int32_t* kept_off,
                   int32_t* n_kept, void* ws);

}  // namespace sp

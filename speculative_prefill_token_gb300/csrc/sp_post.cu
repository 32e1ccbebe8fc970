// Post-processing of the fused SpecPrefill scoring path, after the pool
// kernel has written the pooled scores (W-window mean, llama.cpp PR
// "Speculative prefill" §Approach item 3), their per-tile min / max and the
// per-chunk sums of boost * x and boost.
//
// Both kernels run one CTA per slice of kSliceChunks consecutive chunks of a
// prompt, so a long prompt is spread over many SMs:
//
//   rank    rebuilds every chunk score of the prompt in shared memory --
//           min-max normalisation over the prompt ("SpecPrefill —
//           Implementation Guide" v3.1, item 5), boost x1.5 on the first 64
//           and x1.3 on the last 128 tokens (guide v3, item 2), mean of each
//           32-token chunk (guide §Chunk Selection), taken from the sums
//           because the normalisation is affine -- and decides its own
//           chunks by their position in the order (score descending, chunk
//           index ascending): fixed mode keeps a chunk when fewer than
//           k = max(1, ceil(nc p)) chunks precede it, mass mode when the
//           exact fixed-point sum of the scores preceding it is below
//           ceil(mass * total) (guide v3, item 1: the shortest prefix that
//           reaches the mass, crossing chunk included). The final chunk is
//           forced (PR §Approach item 4). Writes the chunk scores, the keep
//           flags and the slice's kept-token count (chunk 0 counts its BOS
//           token when it is not selected).
//   gather  offsets every slice by the kept tokens of all earlier slices and
//           writes the kept token indices and original positions (guide
//           §How It Works / Sparse Prefill) plus the per-prompt offsets.
//
// The decisions equal those of the radix selection behind sp_select (the
// same set is defined by the same order and threshold, with the same
// float64 and fixed-point arithmetic), and the chunk scores use the same
// operations as the staged chunk kernel, so the fused and the staged paths
// give bit-identical results.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_select.cuh"

namespace sp {
namespace {

constexpr int kRankThreads = 256;
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kWarpChunks = kSliceChunks / kRankWarps;  // chunks ranked by each warp
static_assert(kSliceChunks == 32, "the gather scan uses one lane per chunk of a slice");

struct PostArgs {
    const int32_t* __restrict__ seq_off;
    const int32_t* chunk_off;   // workspace copy
    const int32_t* tile_base;
    const int32_t* slice_base;
    const float2* rpart;        // per pool CTA (128-token tile): (min, max) of the pooled scores
    const float2* __restrict__ csum;  // per chunk (sum boost * x, sum boost)
    float* chunk_score;
    uint8_t* keep;
    int32_t* scount;            // kept tokens per slice
    int32_t* kept_idx;
    int32_t* kept_pos;
    int32_t* kept_off;
    int32_t* n_kept;
    WsHeader* hdr;
    int B, C, mode, normalize, force_bos, force_last;
    float keep_p, mass;
};

__device__ __forceinline__ int64_t chunk_tokens(int64_t n, int C, int64_t c) { return min64(C, n - c * C); }

__global__ void __launch_bounds__(kRankThreads) rank_kernel(const PostArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    if (a.hdr->bad_input) return;
    const int64_t s = blockIdx.x;
    if (s >= a.slice_base[a.B]) return;
    extern __shared__ float cs_s[];  // the prompt's chunk scores
    __shared__ float red_mn[kRankWarps], red_mx[kRankWarps];
    __shared__ unsigned long long red_u[kRankWarps];
    __shared__ float s_mn, s_mx;
    __shared__ unsigned long long s_need;
    __shared__ int s_all, s_S;
    __shared__ int32_t warp_cnt[kRankWarps];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int b = search_base(a.slice_base, a.B, s);
    const int64_t n = static_cast<int64_t>(a.seq_off[b + 1]) - a.seq_off[b];
    const int64_t coff = a.chunk_off[b];
    const int64_t nc = static_cast<int64_t>(a.chunk_off[b + 1]) - coff;
    if (nc > kMaxPromptChunks) {
        // reported; the slice keeps nothing so that the gather stays in bounds
        if (t == 0) {
            atomicCAS(&a.hdr->status, 0, static_cast<int>(SP_ERR_DEVICE));
            a.scount[s] = 0;
        }
        return;
    }
    const int64_t c_lo = (s - a.slice_base[b]) * kSliceChunks;
    const int64_t c_hi = min64(nc, c_lo + kSliceChunks);

    // the first 8 chunk sums of each thread and its tile min / max loads are
    // issued together (one round trip); larger prompts loop
    constexpr int kPre = 8;
    float2 v[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
        const int64_t c = t + k * kRankThreads;
        v[k] = c < nc ? a.csum[coff + c] : make_float2(0.0f, 0.0f);
    }
    // prompt min / max of the pooled scores from the pool kernel's tiles
    float mn = 0.0f, mx = 0.0f;
    if (a.normalize) {
        mn = INFINITY;
        mx = -INFINITY;
        for (int64_t p = a.tile_base[b] + t; p < a.tile_base[b + 1]; p += kRankThreads) {
            const float2 r = a.rpart[p];
            mn = fminf(mn, r.x);
            mx = fmaxf(mx, r.y);
        }
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        if (lane == 0) {
            red_mn[warp] = mn;
            red_mx[warp] = mx;
        }
        __syncthreads();
        if (t == 0) {
            for (int w = 1; w < kRankWarps; ++w) {
                mn = fminf(mn, red_mn[w]);
                mx = fmaxf(mx, red_mx[w]);
            }
            s_mn = mn;
            s_mx = mx;
        }
        __syncthreads();
        mn = s_mn;
        mx = s_mx;
    }
    // every chunk score of the prompt
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
            v[k] = c < nc ? a.csum[coff + c] : make_float2(0.0f, 0.0f);
        }
    }
    const bool is_mass = a.mode == SP_MODE_MASS;
    if (is_mass) {
        for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        if (lane == 0) red_mx[warp] = smax;
    }
    __syncthreads();  // cs_s complete (and the per-warp maxima)
    if (is_mass) {
        if (t == 0) {
            float m = 0.0f;
            for (int w = 0; w < kRankWarps; ++w) m = fmaxf(m, red_mx[w]);
            s_S = mass_scale(nc, m);
        }
        __syncthreads();
        const int S = s_S;
        uint64_t part = 0;
        for (int64_t c = t; c < nc; c += kRankThreads) part += fixed_point(cs_s[c], S);
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red_u[warp] = part;
        __syncthreads();
        if (t == 0) {
            unsigned long long tot = 0;
            for (int w = 0; w < kRankWarps; ++w) tot += red_u[w];
            s_all = tot == 0 ? 1 : 0;
            s_need = mass_threshold(tot, a.mass);
        }
    } else if (t == 0) {
        s_need = fixed_keep_count(nc, a.keep_p);
        s_all = 0;
    }
    __syncthreads();
    const uint64_t need = s_need;
    const bool all = s_all != 0;
    const int S = is_mass ? s_S : 0;

    // warp w ranks chunks c_lo + w + kRankWarps * q of the slice: the count
    // (fixed) or fixed-point mass (mass mode) of the chunks ordered before it.
    // Order key (descending score, ascending index) as one 64-bit integer so
    // that the comparison is branch-free.
    int64_t ci[kWarpChunks];
    uint64_t ki[kWarpChunks];
    uint64_t acc[kWarpChunks];
#pragma unroll
    for (int q = 0; q < kWarpChunks; ++q) {
        ci[q] = c_lo + warp + kRankWarps * q;
        ki[q] = ci[q] < c_hi ? (static_cast<uint64_t>(score_desc_key(cs_s[ci[q]])) << 32) |
                                   static_cast<uint32_t>(ci[q])
                             : 0u;
        acc[q] = 0;
    }
    if (!all) {
        for (int j = lane; j < static_cast<int>(nc); j += 32) {
            const float sj = cs_s[j];
            const uint64_t kj = (static_cast<uint64_t>(score_desc_key(sj)) << 32) | static_cast<uint32_t>(j);
            const uint64_t wj = is_mass ? fixed_point(sj, S) : 1u;
#pragma unroll
            for (int q = 0; q < kWarpChunks; ++q) acc[q] += kj < ki[q] ? wj : 0u;
        }
#pragma unroll
        for (int q = 0; q < kWarpChunks; ++q)
            for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
    }
    if (lane == 0) {
        int32_t my_cnt = 0;
#pragma unroll
        for (int q = 0; q < kWarpChunks; ++q) {
            const int64_t c = ci[q];
            if (c >= c_hi) continue;
            // fixed: fewer than k chunks before it; mass: mass before it below the threshold
            uint8_t f = (all || acc[q] < need) ? 1 : 0;
            if (a.force_last && c == nc - 1) f |= 2;
            a.keep[coff + c] = f;
            my_cnt += static_cast<int32_t>(f ? chunk_tokens(n, a.C, c)
                                             : ((c == 0 && a.force_bos && n > 0) ? 1 : 0));
        }
        warp_cnt[warp] = my_cnt;
    }
    __syncthreads();
    if (t == 0) {
        int32_t tot = 0;
        for (int w = 0; w < kRankWarps; ++w) tot += warp_cnt[w];
        a.scount[s] = tot;
    }
}

// One CTA per slice, plus one past the last slice for the totals.
__global__ void __launch_bounds__(kRankThreads) gather_kernel(const PostArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    if (a.hdr->bad_input) return;
    __shared__ int64_t red[kRankWarps];
    __shared__ int64_t base_s[kSliceChunks];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t S = a.slice_base[a.B];
    const int64_t s = blockIdx.x;
    if (s > S) return;
    // kept tokens of all earlier slices
    int64_t part = 0;
    for (int64_t i = t; i < s; i += kRankThreads) part += a.scount[i];
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[warp] = part;
    __syncthreads();
    int64_t P = 0;
    for (int w = 0; w < kRankWarps; ++w) P += red[w];
    if (s == S) {
        // prompts without tokens at the end of the batch, and the batch total
        if (t == 0) {
            for (int b = a.B - 1; b >= 0 && a.slice_base[b] == S; --b) a.kept_off[b] = static_cast<int32_t>(P);
            a.kept_off[a.B] = static_cast<int32_t>(P);
            *a.n_kept = static_cast<int32_t>(P);
        }
        return;
    }
    const int b = search_base(a.slice_base, a.B, s);
    if (t == 0 && s == a.slice_base[b]) {
        // first slice of prompt b: its offset, and that of empty prompts before it
        for (int bb = b; bb >= 0 && a.slice_base[bb] == s; --bb) a.kept_off[bb] = static_cast<int32_t>(P);
    }
    const int64_t start = a.seq_off[b];
    const int64_t n = static_cast<int64_t>(a.seq_off[b + 1]) - start;
    const int64_t coff = a.chunk_off[b];
    const int64_t nc = static_cast<int64_t>(a.chunk_off[b + 1]) - coff;
    if (nc > kMaxPromptChunks) return;  // reported by the rank kernel; nothing kept
    const int64_t c_lo = (s - a.slice_base[b]) * kSliceChunks;
    // exclusive scan of the slice's per-chunk kept tokens (lane = chunk)
    if (warp == 0) {
        const int64_t c = c_lo + lane;
        int64_t cnt = 0;
        if (c < nc) {
            const uint8_t f = a.keep[coff + c];
            cnt = f ? chunk_tokens(n, a.C, c) : ((c == 0 && a.force_bos && n > 0) ? 1 : 0);
        }
        int64_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        base_s[lane] = P + incl - cnt;
    }
    __syncthreads();
    for (int q = warp; q < kSliceChunks; q += kRankWarps) {
        const int64_t c = c_lo + q;
        if (c >= nc) break;
        const int64_t base = base_s[q];
        if (a.keep[coff + c]) {
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

}  // namespace

cudaError_t launch_post(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                        float* chunk_score, uint8_t* keep, int32_t* kept_idx, int32_t* kept_pos,
                        int32_t* kept_off, int32_t* n_kept, void* ws, cudaStream_t st) {
    PostArgs a;
    a.seq_off = seq_off;
    a.chunk_off = ws_ptr<int32_t>(ws, pl.o_chunk_off);
    a.tile_base = ws_ptr<int32_t>(ws, pl.o_tile_base);
    a.slice_base = ws_ptr<int32_t>(ws, pl.o_slice_base);
    a.rpart = ws_ptr<float2>(ws, pl.o_rpart);
    a.csum = ws_ptr<float2>(ws, pl.o_csum);
    a.chunk_score = chunk_score;
    a.keep = keep;
    a.scount = ws_ptr<int32_t>(ws, pl.o_scount);
    a.kept_idx = kept_idx;
    a.kept_pos = kept_pos;
    a.kept_off = kept_off;
    a.n_kept = n_kept;
    a.hdr = ws_ptr<WsHeader>(ws, 0);
    a.B = pl.B;
    a.C = pl.C;
    a.mode = p->mode;
    a.normalize = p->normalize;
    a.force_bos = p->force_bos;
    a.force_last = p->force_last_chunk;
    a.keep_p = p->keep_p;
    a.mass = p->mass;
    // shared memory for the largest prompt's chunk scores
    const int64_t maxnc = pl.chunks_max < kMaxPromptChunks ? pl.chunks_max : kMaxPromptChunks;
    const size_t smem = static_cast<size_t>(maxnc) * sizeof(float);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const cudaError_t e = launch_k(rank_kernel, static_cast<unsigned>(pl.slices_max), kRankThreads, smem, st, a);
    if (e != cudaSuccess) return e;
    return launch_k(gather_kernel, static_cast<unsigned>(pl.slices_max + 1), kRankThreads, 0, st, a);
}

}  // namespace sp

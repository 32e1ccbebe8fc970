// Per-prompt post-processing of the SpecPrefill scoring path: one CTA per
// prompt, after the pool kernel has written the pooled scores (W-window
// mean, llama.cpp PR "Speculative prefill" §Approach item 3), their per-tile
// min / max and the per-chunk sums.
//
//   normalise  min-max over the prompt ("SpecPrefill — Implementation
//              Guide" v3.1, item 5)
//   boost      x1.5 on the first 64 tokens, x1.3 on the last 128 (guide v3,
//              item 2)
//   chunks     mean of each 32-token chunk (guide §Chunk Selection), from
//              the per-chunk sums of boost * x and boost the pool kernel
//              wrote (the min-max normalisation is affine)
//   select     radix select (sp_select.cuh): top k = max(1, ceil(nc p)) or
//              the shortest prefix holding `mass` of the total (guide v3,
//              item 1); the final chunk and BOS are forced (PR §Approach
//              item 4)
//   offsets    kept tokens per chunk and their scan (the wide gather kernel
//              then writes the kept token indices and original positions,
//              guide §How It Works / Sparse Prefill); the batch offsets come
//              from the last prompt to finish (one prompt: directly).
//
// Every arithmetic step matches the stage kernels behind sp_pool_chunk /
// sp_select / sp_gather_kept operation for operation, so the fused and the
// staged paths give bit-identical results.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_select.cuh"

namespace sp {
namespace {

constexpr int kPostThreads = kSelectThreads;

struct PostArgs {
    const int32_t* __restrict__ seq_off;
    const int32_t* chunk_off;  // workspace copy
    const int32_t* tile_base;
    const float2* rpart;       // per pool CTA (min, max) of the pooled scores
    const float2* __restrict__ csum;  // per chunk (sum boost * x, sum boost)
    float* __restrict__ chunk_score;
    uint8_t* keep;
    int32_t* ckoff;
    int32_t* pcount;
    int32_t* kept_off;
    int32_t* n_kept;
    WsHeader* hdr;
    int B, C, mode, normalize, force_bos, force_last, bf_n, bl_n, rparts_per_tile;
    float keep_p, mass, bf_mult, bl_mult;
};

__device__ __forceinline__ int64_t block_scan_i64(int64_t v, int64_t* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < static_cast<int>(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    const int64_t r = v + (warp > 0 ? warp_tot[warp - 1] : 0);
    __syncthreads();
    return r;
}

// Record the prompt's kept count; with one prompt write the batch offsets
// directly, otherwise the last prompt to finish (ticket) writes kept_off
// and n_kept for the whole batch.
__device__ void finish_batch(const PostArgs& a, int b, int64_t count, int64_t* scan_i) {
    __shared__ int64_t carry;
    __shared__ bool last_prompt;
    const int t = threadIdx.x;
    if (a.B == 1) {
        if (t == 0) {
            a.pcount[0] = static_cast<int32_t>(count);
            a.kept_off[0] = 0;
            a.kept_off[1] = static_cast<int32_t>(count);
            *a.n_kept = static_cast<int32_t>(count);
        }
        return;
    }
    if (t == 0) {
        a.pcount[b] = static_cast<int32_t>(count);
        __threadfence();
        const unsigned prev = atomicAdd(&a.hdr->ticket, 1u);
        last_prompt = (prev == static_cast<unsigned>(a.B - 1));
        carry = 0;
    }
    __syncthreads();
    if (!last_prompt) return;
    __threadfence();
    for (int base = 0; base < a.B; base += kPostThreads) {
        const int bb = base + t;
        const int64_t v = bb < a.B ? static_cast<int64_t>(__ldcg(a.pcount + bb)) : 0;
        const int64_t incl = block_scan_i64(v, scan_i);
        if (bb < a.B) a.kept_off[bb] = static_cast<int32_t>(carry + incl - v);
        __syncthreads();
        if (t == kPostThreads - 1) carry += incl;
        __syncthreads();
    }
    if (t == 0) {
        a.kept_off[a.B] = static_cast<int32_t>(carry);
        *a.n_kept = static_cast<int32_t>(carry);
        a.hdr->ticket = 0u;
    }
}

__global__ void __launch_bounds__(kPostThreads) post_kernel(const PostArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    if (a.hdr->bad_input) return;
    extern __shared__ __align__(16) unsigned char dyn[];
    // [SelectShared][max nc floats: chunk scores][max nc flag bytes]
    SelectShared& ss = *reinterpret_cast<SelectShared*>(dyn);
    float* cs_s = reinterpret_cast<float*>(dyn + ((sizeof(SelectShared) + 15) & ~size_t(15)));
    __shared__ int64_t scan_i[32];
    __shared__ float red_mn[32], red_mx[32];
    __shared__ float s_mn, s_mx;
    __shared__ int64_t carry;
    const int b = blockIdx.x;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t n = static_cast<int64_t>(a.seq_off[b + 1]) - a.seq_off[b];
    const int64_t coff = a.chunk_off[b];
    const int64_t nc = static_cast<int64_t>(a.chunk_off[b + 1]) - coff;
    uint8_t* flags = reinterpret_cast<uint8_t*>(cs_s + kMaxPromptChunks);

    int64_t count = 0;
    if (nc > kMaxPromptChunks) {
        if (t == 0) atomicCAS(&a.hdr->status, 0, static_cast<int>(SP_ERR_DEVICE));
    } else if (nc > 0) {
        // prompt min / max of the pooled scores from the reduce CTAs' partials
        float mn = INFINITY, mx = -INFINITY;
        if (a.normalize) {
            const int64_t p0 = static_cast<int64_t>(a.tile_base[b]) * a.rparts_per_tile;
            const int64_t p1 = static_cast<int64_t>(a.tile_base[b + 1]) * a.rparts_per_tile;
            for (int64_t p = p0 + t; p < p1; p += kPostThreads) {
                const float2 v = a.rpart[p];
                mn = fminf(mn, v.x);
                mx = fmaxf(mx, v.y);
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
                for (int w = 1; w < kPostThreads / 32; ++w) {
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
        // chunk scores from the per-chunk sums (all of a thread's loads first)
        for (int64_t c0 = t; c0 < nc; c0 += kPostThreads * 8) {
            float2 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int64_t c = c0 + k * kPostThreads;
                v[k] = c < nc ? a.csum[coff + c] : make_float2(0.0f, 0.0f);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int64_t c = c0 + k * kPostThreads;
                if (c < nc) {
                    const float cs = chunk_score_from_sums(v[k].x, v[k].y, mn, mx, a.normalize,
                                                           min64(a.C, n - c * a.C));
                    cs_s[c] = cs;
                    a.chunk_score[coff + c] = cs;
                }
            }
        }
        for (int64_t c = t; c < nc; c += kPostThreads) flags[c] = 0;
        __syncthreads();
        radix_select(cs_s, nc, a.mode, a.keep_p, a.mass, flags, ss);
        __syncthreads();
        if (a.force_last && t == 0) flags[nc - 1] |= 2;
        __syncthreads();
        for (int64_t c = t; c < nc; c += kPostThreads) a.keep[coff + c] = flags[c];
        // kept tokens per chunk and their exclusive scan, in chunk order:
        // thread t owns chunks [t*E, t*E + E), one block scan of the totals
        const int64_t E = (nc + kPostThreads - 1) / kPostThreads;
        const int64_t c_lo = min64(nc, static_cast<int64_t>(t) * E), c_hi = min64(nc, c_lo + E);
        int64_t mine = 0;
        for (int64_t c = c_lo; c < c_hi; ++c) {
            const int64_t size = min64(a.C, n - c * a.C);
            mine += flags[c] ? size : ((c == 0 && a.force_bos && n > 0) ? 1 : 0);
        }
        const int64_t incl = block_scan_i64(mine, scan_i);
        int64_t run = incl - mine;
        for (int64_t c = c_lo; c < c_hi; ++c) {
            const int64_t size = min64(a.C, n - c * a.C);
            a.ckoff[coff + c] = static_cast<int32_t>(run);
            run += flags[c] ? size : ((c == 0 && a.force_bos && n > 0) ? 1 : 0);
        }
        if (t == kPostThreads - 1) carry = incl;
        __syncthreads();
        count = carry;
    }
    finish_batch(a, b, count, scan_i);
}

}  // namespace

cudaError_t launch_post(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                        const float* imp, float* tok, float* chunk_score, uint8_t* keep,
                        int32_t* kept_idx, int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept,
                        void* ws, cudaStream_t st) {
    (void)imp;
    PostArgs a;
    a.seq_off = seq_off;
    a.chunk_off = ws_ptr<int32_t>(ws, pl.o_chunk_off);
    a.tile_base = ws_ptr<int32_t>(ws, pl.o_tile_base);
    a.rpart = ws_ptr<float2>(ws, pl.o_rpart);
    a.csum = ws_ptr<float2>(ws, pl.o_csum);
    (void)tok;
    a.chunk_score = chunk_score;
    a.keep = keep;
    a.ckoff = ws_ptr<int32_t>(ws, pl.o_ckoff);
    a.pcount = ws_ptr<int32_t>(ws, pl.o_pcount);
    a.kept_off = kept_off;
    a.n_kept = n_kept;
    (void)kept_idx;
    (void)kept_pos;
    a.hdr = ws_ptr<WsHeader>(ws, 0);
    a.B = pl.B;
    a.C = pl.C;
    a.mode = p->mode;
    a.normalize = p->normalize;
    a.force_bos = p->force_bos;
    a.force_last = p->force_last_chunk;
    a.bf_n = p->boost_first_n;
    a.bl_n = p->boost_last_n;
    a.rparts_per_tile = 1;  // one pool CTA per 128-token tile
    a.keep_p = p->keep_p;
    a.mass = p->mass;
    a.bf_mult = p->boost_first_mult;
    a.bl_mult = p->boost_last_mult;
    const size_t smem = ((sizeof(SelectShared) + 15) & ~size_t(15)) + static_cast<size_t>(kMaxPromptChunks) * 5;
    cudaError_t e = cudaFuncSetAttribute(post_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(post_kernel, static_cast<unsigned>(pl.B), kPostThreads, smem, st, a);
}

}  // namespace sp

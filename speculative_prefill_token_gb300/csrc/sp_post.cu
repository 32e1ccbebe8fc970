// Per-prompt post-processing of the SpecPrefill scoring path in one launch:
// one thread-block cluster of 8 CTAs per prompt.
//
//   pool       x[t] = mean of imp over the centred W-window inside the
//              prompt (llama.cpp PR "Speculative prefill", §Approach item 3)
//   normalise  min-max over the prompt ("SpecPrefill — Implementation
//              Guide" v3.1, item 5); the per-CTA min/max are combined across
//              the cluster through distributed shared memory
//   boost      x1.5 on the first 64 tokens, x1.3 on the last 128 (guide v3,
//              item 2)
//   chunks     mean of each 32-token chunk (guide §Chunk Selection)
//   select     rank 0 runs the radix select of sp_select.cuh: the top
//              k = max(1, ceil(nc p)) chunks or the shortest prefix holding
//              `mass` of the total (guide v3, item 1); the final chunk and BOS
//              are forced (PR §Approach item 4)
//   gather     kept token indices and original positions (guide §How It
//              Works / Sparse Prefill), written by every rank for its own
//              chunks when the batch has one prompt; with several prompts
//              the last prompt to finish writes the batch offsets and a
//              separate gather kernel writes the lists.
//
// The arithmetic of every step matches the stage kernels of sp_pool_chunk /
// sp_select / sp_gather_kept operation for operation, so the fused and the
// staged paths give bit-identical results.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_select.cuh"

namespace cg = cooperative_groups;

namespace sp {
namespace {

constexpr int kCluster = 8;
constexpr int kPostThreads = 1024;

struct PostArgs {
    const int32_t* seq_off;
    const int32_t* chunk_off;  // workspace copy
    const float* imp;
    float* tok;
    float* chunk_score;
    uint8_t* keep;
    int32_t* ckoff;
    int32_t* pcount;
    int32_t* kept_off;
    int32_t* n_kept;
    int32_t* kept_idx;
    int32_t* kept_pos;
    WsHeader* hdr;
    int B, C, W, mode, normalize, force_bos, force_last, bf_n, bl_n, write_lists;
    int64_t xs_cap;  // pooled scores of one rank kept in shared memory (0: re-read from tok)
    float keep_p, mass, bf_mult, bl_mult;
};

constexpr int kPrefetch = 8;  // global loads a thread issues before it uses any

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

// Rank 0: selection, forced final chunk, flags, kept tokens per chunk and
// their scan. Returns the prompt's kept-token count.
__device__ int64_t select_prompt(const PostArgs& a, int64_t coff, int64_t nc, int64_t n,
                                 uint8_t* flags, SelectShared& ss) {
    __shared__ int64_t scan_i[32];
    __shared__ int64_t carry;
    const int t = threadIdx.x;
    for (int64_t i = t; i < nc; i += kPostThreads) flags[i] = 0;
    __syncthreads();
    radix_select(a.chunk_score + coff, nc, a.mode, a.keep_p, a.mass, flags, ss);
    __syncthreads();
    if (a.force_last && t == 0) flags[nc - 1] |= 2;
    if (t == 0) carry = 0;
    __syncthreads();
    for (int64_t i = t; i < nc; i += kPostThreads) a.keep[coff + i] = flags[i];
    // kept tokens per chunk and their exclusive scan, in chunk order
    for (int64_t base = 0; base < nc; base += kPostThreads) {
        const int64_t c = base + t;
        int64_t cnt = 0;
        if (c < nc) {
            const int64_t size = min64(a.C, n - c * a.C);
            cnt = flags[c] ? size : ((c == 0 && a.force_bos && n > 0) ? 1 : 0);
        }
        const int64_t incl = block_scan_i64(cnt, scan_i);
        if (c < nc) a.ckoff[coff + c] = static_cast<int32_t>(carry + incl - cnt);
        __syncthreads();
        if (t == kPostThreads - 1) carry += incl;
        __syncthreads();
    }
    return carry;  // read after the loop's closing barrier
}

// Rank 0: record the prompt's kept count; with one prompt write the batch
// offsets directly, otherwise the last prompt to finish (ticket) writes
// kept_off and n_kept for the whole batch.
__device__ void finish_batch(const PostArgs& a, int b, int64_t count) {
    __shared__ int64_t scan_i[32];
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

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kPostThreads)
    post_kernel(const PostArgs a) {
    if (a.hdr->bad_input) return;  // uniform over the grid: no cluster barrier is left waiting
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ float dyn[];  // [TB + 2h] staging | [xs_cap] pooled scores | flags
    __shared__ float red_mn[32], red_mx[32];
    __shared__ float cl_mm[2];
    __shared__ float s_mn, s_mx;
    __shared__ SelectShared ss;
    const int q = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.x / kCluster;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t start = a.seq_off[b];
    const int64_t n = static_cast<int64_t>(a.seq_off[b + 1]) - start;
    const int64_t coff = a.chunk_off[b];
    const int64_t nc = static_cast<int64_t>(a.chunk_off[b + 1]) - coff;
    const int64_t cq0 = nc * q / kCluster, cq1 = nc * (q + 1) / kCluster;
    const int64_t t0 = cq0 * a.C, t1 = min64(cq1 * a.C, n);
    const int h = a.W / 2;
    // staging blocks of TB tokens (a whole number of chunks)
    const int64_t TB = a.C <= 4096 ? static_cast<int64_t>(a.C) * (4096 / a.C) : a.C;
    float* stage = dyn;
    float* xs = dyn + TB + 2 * h;
    const bool keep_x = (t1 - t0) <= a.xs_cap;
    uint8_t* flags = reinterpret_cast<uint8_t*>(xs + a.xs_cap);

    // pass 1: pooled scores of this rank's tokens, and their min / max
    float mn = INFINITY, mx = -INFINITY;
    for (int64_t blk = t0; blk < t1; blk += TB) {
        const int64_t b1 = min64(blk + TB, t1);
        const int64_t lo = max64(0, blk - h), hi = min64(n, b1 + h);
        for (int64_t u0 = lo; u0 < hi; u0 += kPostThreads * kPrefetch) {
            float r[kPrefetch];
#pragma unroll
            for (int k = 0; k < kPrefetch; ++k) {
                const int64_t u = u0 + t + k * kPostThreads;
                r[k] = u < hi ? a.imp[start + u] : 0.0f;
            }
#pragma unroll
            for (int k = 0; k < kPrefetch; ++k) {
                const int64_t u = u0 + t + k * kPostThreads;
                if (u < hi) stage[u - lo] = r[k];
            }
        }
        __syncthreads();
        for (int64_t tt = blk + t; tt < b1; tt += kPostThreads) {
            const int64_t u0 = max64(0, tt - h), u1 = min64(n - 1, tt + h);
            float s = 0.0f;
            for (int64_t u = u0; u <= u1; ++u) s += stage[u - lo];
            const float x = s / static_cast<float>(u1 - u0 + 1);
            a.tok[start + tt] = x;
            if (keep_x) xs[tt - t0] = x;
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
        __syncthreads();
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
        cl_mm[0] = mn;
        cl_mm[1] = mx;
    }
    cluster.sync();
    if (t == 0) {
        float gmn = INFINITY, gmx = -INFINITY;
        for (int r = 0; r < kCluster; ++r) {
            const float* other = cluster.map_shared_rank(cl_mm, r);
            gmn = fminf(gmn, other[0]);
            gmx = fmaxf(gmx, other[1]);
        }
        s_mn = gmn;
        s_mx = gmx;
    }
    __syncthreads();

    // pass 2: normalise, boost and average this rank's chunks
    const float gmn = s_mn, gmx = s_mx;
    for (int64_t blk = t0; blk < t1; blk += TB) {
        const int64_t b1 = min64(blk + TB, t1);
        float* ys = keep_x ? xs + (blk - t0) : stage;
        if (!keep_x) {
            for (int64_t u0 = blk; u0 < b1; u0 += kPostThreads * kPrefetch) {
                float r[kPrefetch];
#pragma unroll
                for (int k = 0; k < kPrefetch; ++k) {
                    const int64_t u = u0 + t + k * kPostThreads;
                    r[k] = u < b1 ? a.tok[start + u] : 0.0f;
                }
#pragma unroll
                for (int k = 0; k < kPrefetch; ++k) {
                    const int64_t u = u0 + t + k * kPostThreads;
                    if (u < b1) ys[u - blk] = r[k];
                }
            }
            __syncthreads();
        }
        for (int64_t tt = blk + t; tt < b1; tt += kPostThreads) {
            float y = ys[tt - blk];
            if (a.normalize) y = (gmx == gmn) ? 1.0f : (y - gmn) / (gmx - gmn);
            if (tt < a.bf_n) y *= a.bf_mult;
            if (tt >= n - a.bl_n) y *= a.bl_mult;
            ys[tt - blk] = y;
        }
        __syncthreads();
        const int64_t c_lo = blk / a.C, c_hi = (b1 + a.C - 1) / a.C;
        for (int64_t c = c_lo + t; c < c_hi; c += kPostThreads) {
            const int64_t a0 = c * a.C, a1 = min64(b1, a0 + a.C);
            float s = 0.0f;
            for (int64_t tt = a0; tt < a1; ++tt) s += ys[tt - blk];
            a.chunk_score[coff + c] = s / static_cast<float>(a1 - a0);
        }
        __syncthreads();
    }
    cluster.sync();  // chunk scores of all ranks visible (cluster-scope release / acquire)

    if (q == 0) {
        int64_t count = 0;
        if (nc > kMaxPromptChunks) {
            if (t == 0) atomicCAS(&a.hdr->status, 0, static_cast<int>(SP_ERR_DEVICE));
        } else if (nc > 0) {
            count = select_prompt(a, coff, nc, n, flags, ss);
        }
        finish_batch(a, b, count);
    }
    if (!a.write_lists) return;  // several prompts: the gather kernel writes the lists
    cluster.sync();  // flags and per-chunk offsets of rank 0 visible
    // this rank's chunks: flags and offsets prefetched, then one warp per chunk
    int32_t* off_s = reinterpret_cast<int32_t*>(stage);
    uint8_t* flg_s = reinterpret_cast<uint8_t*>(off_s + (cq1 - cq0));
    for (int64_t c = cq0 + t; c < cq1; c += kPostThreads) {
        off_s[c - cq0] = a.ckoff[coff + c];
        flg_s[c - cq0] = a.keep[coff + c];
    }
    __syncthreads();
    for (int64_t c = cq0 + warp; c < cq1; c += kPostThreads / 32) {
        const int64_t base = off_s[c - cq0];
        if (flg_s[c - cq0]) {
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
                        const float* imp, float* tok, float* chunk_score, uint8_t* keep,
                        int32_t* kept_idx, int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept,
                        void* ws, cudaStream_t st) {
    PostArgs a;
    a.seq_off = seq_off;
    a.chunk_off = ws_ptr<int32_t>(ws, pl.o_chunk_off);
    a.imp = imp;
    a.tok = tok;
    a.chunk_score = chunk_score;
    a.keep = keep;
    a.ckoff = ws_ptr<int32_t>(ws, pl.o_ckoff);
    a.pcount = ws_ptr<int32_t>(ws, pl.o_pcount);
    a.kept_off = kept_off;
    a.n_kept = n_kept;
    a.kept_idx = kept_idx;
    a.kept_pos = kept_pos;
    a.hdr = ws_ptr<WsHeader>(ws, 0);
    a.B = pl.B;
    a.C = pl.C;
    a.W = p->pool_w;
    a.mode = p->mode;
    a.normalize = p->normalize;
    a.force_bos = p->force_bos;
    a.force_last = p->force_last_chunk;
    a.bf_n = p->boost_first_n;
    a.bl_n = p->boost_last_n;
    a.write_lists = pl.B == 1 ? 1 : 0;
    a.keep_p = p->keep_p;
    a.mass = p->mass;
    a.bf_mult = p->boost_first_mult;
    a.bl_mult = p->boost_last_mult;
    // shared memory: staging block with halo, this rank's pooled scores when
    // they fit, one flag byte per chunk of the prompt (rank 0)
    const int64_t tb = pl.C <= 4096 ? static_cast<int64_t>(pl.C) * (4096 / pl.C) : pl.C;
    const int64_t stage_floats = tb + 2 * (p->pool_w / 2);
    const int64_t max_nc = (pl.Ntot + pl.C - 1) / pl.C < kMaxPromptChunks ? (pl.Ntot + pl.C - 1) / pl.C
                                                                          : kMaxPromptChunks;
    const int64_t rank_tokens = ((max_nc + kCluster - 1) / kCluster) * pl.C;
    const int64_t budget = (200 << 10) / 4 - stage_floats - (max_nc + 3) / 4;
    a.xs_cap = rank_tokens <= budget ? rank_tokens : (budget > 0 ? budget : 0);
    const size_t smem = sizeof(float) * static_cast<size_t>(stage_floats + a.xs_cap) +
                        static_cast<size_t>(max_nc) + 16;
    cudaError_t e = cudaFuncSetAttribute(post_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    post_kernel<<<static_cast<unsigned>(pl.B * kCluster), kPostThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace sp

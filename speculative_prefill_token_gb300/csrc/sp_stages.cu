// Stage kernels of the SpecPrefill scoring path after (and around) the
// logits: per-call offsets, softmax normalisers, token importance, pooling,
// chunk scores, selection and the kept-token gather.
//
// Method steps (pages: "SpecPrefill — Implementation Guide" v2/v3.1 of the
// sliding-specprefill project; llama.cpp PR "Speculative prefill"):
//   normaliser + importance  guide §How It Works / Token Importance
//   pool (W = 13)            PR §Approach item 3
//   normalise                guide v3.1 §v3.1 Optimizations item 5
//   boost                    guide v3 §v3 Improvements item 2
//   chunk mean, ranking      guide §Chunk Selection
//   cumulative mass          guide v3 §v3 Improvements item 1
//   forced BOS / last chunk  PR §Approach item 4
//   kept list + positions    guide §How It Works / Sparse Prefill
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_phases.cuh"
#include "sp_select.cuh"

namespace sp {
namespace {

__device__ __forceinline__ void set_status(WsHeader* h, int code) { atomicCAS(&h->status, 0, code); }

// ------------------------------------------------------------------ prep
// One CTA: validates seq_off (0 = first, non-decreasing, last = Ntot, no
// prompt longer than the shape's max_seq_len when that is set) and
// writes the per-prompt bases of logits tiles, chunks and post blocks.
// A user-provided chunk_off (standalone select/gather) must match.
constexpr int kPrepThreads = 256;  // small enough to share an SM with the logits kernel

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const int32_t* seq_off, int B,
                                                            int64_t Ntot, int C, int64_t Tb,
                                                            int32_t* tile_base, int32_t* chunk_off,
                                                            int32_t* pblk_base, int32_t* slice_base,
                                                            int32_t* chunk_off_out,
                                                            const int32_t* chunk_off_check,
                                                            unsigned* seg_cnt, int64_t n_seg_cnt,
                                                            int block_size, int table_stride,
                                                            int max_len, WsHeader* hdr) {
    grid_dep_wait();
    grid_dep_launch();
    __shared__ int bad;
    __shared__ int64_t warp_sums[4][32];
    const int tid = threadIdx.x;
    if (tid == 0) {
        bad = (seq_off[0] != 0 || static_cast<int64_t>(seq_off[B]) != Ntot) ? 1 : 0;
        hdr->ticket = 0u;
    }
    __syncthreads();
    for (int b = tid; b < B; b += kPrepThreads) {
        const int64_t n = static_cast<int64_t>(seq_off[b + 1]) - seq_off[b];
        if (n < 0) bad = 1;
        // a prompt longer than the caller's stated bound
        if (max_len > 0 && n > max_len) bad = 1;
        // a block-paged key source must list every block of the prompt
        if (block_size > 0 && (n + block_size - 1) / block_size > table_stride) bad = 1;
    }
    for (int64_t i = tid; i < n_seg_cnt; i += kPrepThreads) seg_cnt[i] = 0u;
    __syncthreads();
    const int per = (B + kPrepThreads - 1) / kPrepThreads;
    const int lo = min(B, tid * per), hi = min(B, lo + per);
    int64_t sums[4] = {0, 0, 0, 0};
    if (!bad) {
        for (int b = lo; b < hi; ++b) {
            const int64_t n = static_cast<int64_t>(seq_off[b + 1]) - seq_off[b];
            sums[0] += (n + kTileTokens - 1) / kTileTokens;
            sums[1] += (n + C - 1) / C;
            sums[2] += (n + Tb - 1) / Tb;
            sums[3] += ((n + C - 1) / C + kSliceChunks - 1) / kSliceChunks;
        }
    }
    // block exclusive scan of the three per-thread totals
    const int lane = tid & 31, warp = tid >> 5;
    int64_t incl[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        int64_t v = sums[k];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        incl[k] = v;
        if (lane == 31) warp_sums[k][warp] = v;
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            int64_t v = warp_sums[k][lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            warp_sums[k][lane] = v;  // inclusive over warps
        }
    }
    __syncthreads();
    int64_t run[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) run[k] = incl[k] - sums[k] + (warp > 0 ? warp_sums[k][warp - 1] : 0);
    for (int b = lo; b < hi; ++b) {
        const int64_t n = bad ? 0 : static_cast<int64_t>(seq_off[b + 1]) - seq_off[b];
        tile_base[b] = static_cast<int32_t>(run[0]);
        chunk_off[b] = static_cast<int32_t>(run[1]);
        pblk_base[b] = static_cast<int32_t>(run[2]);
        slice_base[b] = static_cast<int32_t>(run[3]);
        if (chunk_off_out) chunk_off_out[b] = static_cast<int32_t>(run[1]);
        if (chunk_off_check && chunk_off_check[b] != static_cast<int32_t>(run[1])) bad = 1;
        run[0] += (n + kTileTokens - 1) / kTileTokens;
        run[1] += (n + C - 1) / C;
        run[2] += (n + Tb - 1) / Tb;
        run[3] += ((n + C - 1) / C + kSliceChunks - 1) / kSliceChunks;
    }
    if (hi == B && lo < hi) {
        tile_base[B] = static_cast<int32_t>(run[0]);
        chunk_off[B] = static_cast<int32_t>(run[1]);
        pblk_base[B] = static_cast<int32_t>(run[2]);
        slice_base[B] = static_cast<int32_t>(run[3]);
        if (chunk_off_out) chunk_off_out[B] = static_cast<int32_t>(run[1]);
        if (chunk_off_check && chunk_off_check[B] != static_cast<int32_t>(run[1])) bad = 1;
    }
    __syncthreads();
    if (tid == 0) {
        hdr->bad_input = bad;
        if (bad) set_status(hdr, SP_ERR_DEVICE);
    }
}

// --------------------------------------------------------------- reduce
// Token importance from the wave's quantised logits. One CTA covers TOK =
// 1024 / Rs tokens of one tile (Rs / 8 threads per token, 8 rows each):
// every thread loads its eight 16-bit values of every slab (16 bytes,
// coalesced) and keeps the max over slabs of
// y - lse2 = (M - lse2) - q / kLogitQuant, the log2 softmax probability,
// with M - lse2 taken from a per-CTA table [warp quarter][slab][row]. The
// max over the G heads of each lookahead step is then combined with earlier
// waves and (last wave) imp[t] = (1/L) sum_l exp2(max over layers, heads)
// written: when G divides 8, by the token's own threads from registers
// (their partial sums added by shuffles; 2B workload 62.6 -> 62.1 us per
// call, 0.8B 34.7 -> 33.9, serving batch 240.8 -> 238.5), else by one
// thread per token through shared memory (kFast: the former, a separate
// instance without the latter's registers, which lets six slabs per thread
// be in flight without spills: long workload 243.2 -> 241.1, serving 238.3
// -> 237.3, 2B unchanged). Small CTAs (eight per SM) spread a wave over
// every SM that the logits kernel frees.
constexpr int kReduceThreads = 128;
constexpr int kReduceSlabBatch = 6;

template <bool kFast>
__global__ void __launch_bounds__(kReduceThreads, 8) reduce_kernel(
    const uint16_t* logits, const float* lmax, const float* lse2, const int32_t* seq_off,
    const int32_t* tile_base, float* alog, float* imp, int B, int G, int L, int R, int Rs, int nslab,
    int64_t Ntot, int64_t rows_per_slab, int64_t tiles_max, int first_wave, int last_wave,
    const int32_t* bad) {
    grid_dep_wait();   // no early release: the pool kernel spreads over every SM once this one ends
    const int Q8 = Rs / 8;
    const int TOK = kReduceThreads / Q8;
    const int subs = kTileTokens / TOK;
    const int64_t tile = blockIdx.x / subs;
    const int sub = blockIdx.x - static_cast<int>(tile) * subs;
    const int tq = threadIdx.x / Q8, c = threadIdx.x - tq * Q8;
    const int64_t row = tile * kTileTokens + static_cast<int64_t>(sub) * TOK + tq;
    const uint4* src = reinterpret_cast<const uint4*>(logits + row * Rs + 8 * c);
    const int64_t slab_stride = rows_per_slab * Rs / 8;  // in 16-byte units
    // the first batch depends on the block index only (every tile slot of the
    // scratch exists), so it is requested before the offsets and maxima;
    // later batches while the current one is reduced
    uint4 v[kReduceSlabBatch];
#pragma unroll
    for (int u = 0; u < kReduceSlabBatch; ++u)
        if (u < nslab) v[u] = __ldcs(src + u * slab_stride);
    extern __shared__ float sm[];
    const int q0 = sub * TOK / 32, nq = (TOK + 31) / 32;  // warp quarters of the CTA's tokens
    float* off_s = sm;                       // [nq][nslab][Rs]: M - lse2
    float* ms = off_s + nq * nslab * Rs;     // [TOK][Rs + 1]
    // A single prompt (B = 1) has seq_off = {0, Ntot} once the prep kernel
    // has accepted the input: its offsets come from Ntot and the table is
    // requested before the flag is read.
    const auto fill_table = [&](int b) {
        for (int idx = threadIdx.x; idx < nq * nslab * Rs; idx += kReduceThreads) {
            const int qq = idx / (nslab * Rs), rem = idx - qq * nslab * Rs;
            const int s = rem / Rs, r = rem - s * Rs;
            off_s[idx] = lmax[((static_cast<int64_t>(s) * tiles_max + tile) * 4 + q0 + qq) * Rs + r] -
                         lse2[(static_cast<int64_t>(s) * B + b) * Rs + r];
        }
    };
    const bool one = B == 1;
    int b = 0;
    int64_t i, start, n;
    if (one) {
        if (tile >= (Ntot + kTileTokens - 1) / kTileTokens) return;
        fill_table(0);
        if (*bad) return;
        i = tile;
        start = 0;
        n = Ntot;
    } else {
        const int32_t* const aux[1] = {seq_off};
        const int32_t bad_v = *bad;
        const Located<1> loc = locate<1>(tile_base, aux, B, tile);
        if (bad_v) return;
        if (tile >= loc.total) return;
        b = loc.b;
        i = tile - loc.base_b;
        start = loc.lo[0];
        n = static_cast<int64_t>(loc.hi[0]) - start;
    }
    const int64_t first = i * kTileTokens + static_cast<int64_t>(sub) * TOK;  // within the prompt
    const int nvalid = static_cast<int>(min64(TOK, n - first));
    if (nvalid <= 0) return;
    const bool act = tq < nvalid;
    if (!one) fill_table(b);
    __syncthreads();
    const float* ot = off_s + (tq / 32) * nslab * Rs + 8 * c;  // this token's quarter
    float m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = -INFINITY;
    for (int s0 = 0; s0 < nslab; s0 += kReduceSlabBatch) {
#pragma unroll
        for (int u = 0; u < kReduceSlabBatch; ++u) {
            if (act && s0 + u < nslab) {
                const float* os = ot + (s0 + u) * Rs;
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    m[2 * k] = fmaxf(m[2 * k], fmaf(-static_cast<float>(w[k] & 0xffffu), kLogitQuantInv, os[2 * k]));
                    m[2 * k + 1] = fmaxf(m[2 * k + 1], fmaf(-static_cast<float>(w[k] >> 16), kLogitQuantInv, os[2 * k + 1]));
                }
            }
        }
        const int s1 = s0 + kReduceSlabBatch;
#pragma unroll
        for (int u = 0; u < kReduceSlabBatch; ++u)
            if (act && s1 + u < nslab) v[u] = __ldcs(src + (s1 + u) * slab_stride);
    }
    if (kFast) {  // G divides 8
        // each thread's eight rows are 8 / G whole lookahead steps (row =
        // step * G + head): their head maxima stay in registers, and the
        // Q8 threads of a token (adjacent lanes) add their terms by shuffles
        float gm[8];
        int ng = 0;
        if (G == 1) {
#pragma unroll
            for (int k = 0; k < 8; ++k) gm[k] = m[k];
            ng = 8;
        } else if (G == 2) {
#pragma unroll
            for (int k = 0; k < 4; ++k) gm[k] = fmaxf(m[2 * k], m[2 * k + 1]);
            ng = 4;
        } else if (G == 4) {
#pragma unroll
            for (int k = 0; k < 2; ++k) gm[k] = fmaxf(fmaxf(m[4 * k], m[4 * k + 1]), fmaxf(m[4 * k + 2], m[4 * k + 3]));
            ng = 2;
        } else {
            gm[0] = fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
            ng = 1;
        }
        float part = 0.0f;
        const int64_t tok = start + first + tq;
        const int l0 = 8 * c / G;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k < ng && act && l0 + k < L) {
                const int l = l0 + k;
                float a = gm[k];
                if (!first_wave) a = fmaxf(a, alog[l * Ntot + tok]);
                if (last_wave) part += exp2f(a);
                else alog[l * Ntot + tok] = a;
            }
        }
        if (last_wave) {
            for (int o = 1; o < Q8; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (act && c == 0) imp[tok] = part / static_cast<float>(L);
        }
        return;
    }
    if (act) {
        float* mrow = ms + tq * (Rs + 1) + 8 * c;
#pragma unroll
        for (int k = 0; k < 8; ++k) mrow[k] = m[k];
    }
    __syncthreads();
    const int t = threadIdx.x;
    if (t < nvalid) {
        const int64_t tok = start + first + t;
        const float* mrow = ms + t * (Rs + 1);
        float total = 0.0f;
        for (int l = 0; l < L; ++l) {
            float a = -INFINITY;
            for (int j = 0; j < G; ++j) a = fmaxf(a, mrow[l * G + j]);
            if (!first_wave) a = fmaxf(a, alog[l * Ntot + tok]);
            if (last_wave) total += exp2f(a);
            else alog[l * Ntot + tok] = a;
        }
        if (last_wave) imp[tok] = total / static_cast<float>(L);
    }
}

// --------------------------------------------------------- pool + chunk sums
// Fused-path pooling: one CTA per 128-token tile of a prompt (pool_tile).
__global__ void __launch_bounds__(kPoolThreads) pool_sums_kernel(const PoolArgs a, const int32_t* bad) {
    grid_dep_wait();   // no early release (see the rank kernel)
    const int64_t tile = blockIdx.x;
    __shared__ PoolShared sh;
    if (a.B == 1) {  // pool_tile reads the flag after requesting the window
        const int64_t hi[2] = {a.Ntot, (a.Ntot + a.C - 1) / a.C};
        const Located<2> loc = one_prompt<2>(static_cast<int32_t>((a.Ntot + kTileTokens - 1) / kTileTokens), hi);
        if (tile >= loc.total) return;
        pool_tile(a, tile, threadIdx.x, GroupBar{1, kPoolThreads}, sh, loc, bad);
        return;
    }
    const int32_t* const aux[2] = {a.seq_off, a.chunk_off};
    const int32_t bad_v = *bad;
    const Located<2> loc = locate<2>(a.tile_base, aux, a.B, tile);
    if (bad_v) return;
    if (tile >= loc.total) return;
    pool_tile(a, tile, threadIdx.x, GroupBar{1, kPoolThreads}, sh, loc, nullptr);
}

// ----------------------------------------------------------------- pool
// x[t] = mean of imp over [t - W/2, t + W/2] clipped to the prompt; per
// block min/max of x for the normalisation.
__global__ void __launch_bounds__(256) pool_kernel(const float* imp, float* tok, float2* ppart,
                                                   const int32_t* seq_off, const int32_t* pblk_base,
                                                   int B, int W, int64_t Tb, const int32_t* bad) {
    grid_dep_wait();
    grid_dep_launch();
    if (*bad) return;
    const int64_t blk = blockIdx.x;
    if (blk >= pblk_base[B]) return;
    extern __shared__ float win[];
    __shared__ float red_min[8], red_max[8];
    const int b = search_base(pblk_base, B, blk);
    const int64_t i = blk - pblk_base[b];
    const int64_t start = seq_off[b];
    const int64_t n = static_cast<int64_t>(seq_off[b + 1]) - start;
    const int64_t t0 = i * Tb, t1 = min64(n, t0 + Tb);
    const int h = W / 2;
    const int64_t lo = max64(0, t0 - h), hi = min64(n, t1 + h);
    for (int64_t u = lo + threadIdx.x; u < hi; u += blockDim.x) win[u - lo] = imp[start + u];
    __syncthreads();
    float mn = INFINITY, mx = -INFINITY;
    for (int64_t t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
        const int64_t u0 = max64(0, t - h), u1 = min64(n - 1, t + h);
        float s = 0.0f;
        for (int64_t u = u0; u <= u1; ++u) s += win[u - lo];
        const float x = s / static_cast<float>(u1 - u0 + 1);
        tok[start + t] = x;
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
    }
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red_min[warp] = mn;
        red_max[warp] = mx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
            mn = fminf(mn, red_min[w]);
            mx = fmaxf(mx, red_max[w]);
        }
        ppart[blk] = make_float2(mn, mx);
    }
}

// ---------------------------------------------------------------- chunk
// y = normalise(x) (optional) then boost, and the mean of y over each
// chunk of the block.
__global__ void __launch_bounds__(256) chunk_kernel(const float* tok, const float2* ppart,
                                                    float* chunk_score, const int32_t* seq_off,
                                                    const int32_t* pblk_base, const int32_t* chunk_off,
                                                    int B, int C, int64_t Tb, int normalize,
                                                    float bf_mult, int bf_n, float bl_mult, int bl_n,
                                                    const int32_t* bad) {
    grid_dep_wait();
    grid_dep_launch();
    if (*bad) return;
    const int64_t blk = blockIdx.x;
    if (blk >= pblk_base[B]) return;
    extern __shared__ float ys[];
    __shared__ float red_min[8], red_max[8];
    __shared__ float s_mn, s_mx;
    const int b = search_base(pblk_base, B, blk);
    const int64_t i = blk - pblk_base[b];
    const int64_t start = seq_off[b];
    const int64_t n = static_cast<int64_t>(seq_off[b + 1]) - start;
    const int64_t t0 = i * Tb, t1 = min64(n, t0 + Tb);
    if (normalize) {
        float mn = INFINITY, mx = -INFINITY;
        for (int64_t p = pblk_base[b] + threadIdx.x; p < pblk_base[b + 1]; p += blockDim.x) {
            const float2 v = ppart[p];
            mn = fminf(mn, v.x);
            mx = fmaxf(mx, v.y);
        }
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (lane == 0) {
            red_min[warp] = mn;
            red_max[warp] = mx;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
                mn = fminf(mn, red_min[w]);
                mx = fmaxf(mx, red_max[w]);
            }
            s_mn = mn;
            s_mx = mx;
        }
        __syncthreads();
    }
    const float mn = normalize ? s_mn : 0.0f, mx = normalize ? s_mx : 0.0f;
    for (int64_t t = t0 + threadIdx.x; t < t1; t += blockDim.x) ys[t - t0] = tok[start + t];
    __syncthreads();
    // one warp per chunk, in the order of the fused path's pool kernel
    const int64_t c0 = t0 / C, c1 = (t1 + C - 1) / C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t c = c0 + warp; c < c1; c += blockDim.x >> 5) {
        const int64_t a0 = c * C, a1 = min64(t1, a0 + C);
        const float2 r = warp_chunk_sums(ys, t0, a0, a1, n, bf_n, bf_mult, bl_n, bl_mult, lane);
        if (lane == 0) chunk_score[chunk_off[b] + c] = chunk_score_from_sums(r.x, r.y, mn, mx, normalize, a1 - a0);
    }
}

// --------------------------------------------------------------- select
constexpr int kSelThreads = kSelectThreads;

// Block-wide inclusive scan of one int64 per thread.
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
        int64_t w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
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

// Per-prompt kept-token counts of each chunk, their exclusive scan, the
// prompt's total; the last prompt to finish (ticket) writes kept_off and
// n_kept for the whole batch.
__device__ void scan_kept(const uint8_t* flags, int64_t nc, int64_t n, int C, int force_bos, int b,
                          int B, int32_t* ckoff, int32_t* pcount, int32_t* kept_off,
                          int32_t* n_kept, WsHeader* hdr, int64_t* scratch) {
    __shared__ int64_t carry;
    __shared__ bool last;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < nc; base += blockDim.x) {
        const int64_t c = base + threadIdx.x;
        int64_t cnt = 0;
        if (c < nc) {
            const int64_t size = min64(C, n - c * C);
            cnt = flags[c] ? size : ((c == 0 && force_bos && n > 0) ? 1 : 0);
        }
        const int64_t incl = block_scan_i64(cnt, scratch);
        if (c < nc) ckoff[c] = static_cast<int32_t>(carry + incl - cnt);
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry += incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        pcount[b] = static_cast<int32_t>(carry);
        __threadfence();
        const unsigned prev = atomicAdd(&hdr->ticket, 1u);
        last = (prev == static_cast<unsigned>(B - 1));
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < B; base += blockDim.x) {
        const int bb = base + threadIdx.x;
        const int64_t v = bb < B ? static_cast<int64_t>(__ldcg(pcount + bb)) : 0;
        const int64_t incl = block_scan_i64(v, scratch);
        if (bb < B) kept_off[bb] = static_cast<int32_t>(carry + incl - v);
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry += incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        kept_off[B] = static_cast<int32_t>(carry);
        *n_kept = static_cast<int32_t>(carry);
        hdr->ticket = 0u;
    }
}

// One CTA per prompt: radix selection, then the forced final chunk.
__global__ void __launch_bounds__(kSelThreads) select_kernel(const int32_t* chunk_off,
                                                             const float* chunk_score,
                                                             uint8_t* keep, WsHeader* hdr, int mode,
                                                             float keep_p, float mass,
                                                             int force_last) {
    grid_dep_wait();
    grid_dep_launch();
    if (hdr->bad_input) return;
    extern __shared__ __align__(16) unsigned char dyn[];
    SelectShared& ss = *reinterpret_cast<SelectShared*>(dyn);
    float* sc_s = reinterpret_cast<float*>(dyn + ((sizeof(SelectShared) + 15) & ~size_t(15)));
    uint8_t* flags = reinterpret_cast<uint8_t*>(sc_s + kMaxPromptChunks);
    const int b = blockIdx.x;
    const int64_t c0 = chunk_off[b];
    const int64_t nc = static_cast<int64_t>(chunk_off[b + 1]) - c0;
    if (nc > kMaxPromptChunks) {
        if (threadIdx.x == 0) atomicCAS(&hdr->status, 0, static_cast<int>(SP_ERR_DEVICE));
        return;
    }
    if (nc == 0) return;
    for (int64_t i = threadIdx.x; i < nc; i += kSelThreads) {
        flags[i] = 0;
        sc_s[i] = chunk_score[c0 + i];
    }
    __syncthreads();
    radix_select(sc_s, nc, mode, keep_p, mass, flags, ss);
    __syncthreads();
    if (force_last && threadIdx.x == 0) flags[nc - 1] |= 2;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < nc; i += kSelThreads) keep[c0 + i] = flags[i];
}

__global__ void __launch_bounds__(kSelThreads) gather_scan_kernel(
    const int32_t* seq_off, const int32_t* chunk_off, const uint8_t* keep, int32_t* ckoff,
    int32_t* pcount, int32_t* kept_off, int32_t* n_kept, WsHeader* hdr, int B, int C,
    int force_bos) {
    grid_dep_wait();
    grid_dep_launch();
    if (hdr->bad_input) return;
    __shared__ int64_t scan_i[32];
    const int b = blockIdx.x;
    const int64_t c0 = chunk_off[b];
    const int64_t nc = static_cast<int64_t>(chunk_off[b + 1]) - c0;
    const int64_t n = static_cast<int64_t>(seq_off[b + 1]) - seq_off[b];
    scan_kept(keep + c0, nc, n, C, force_bos, b, B, ckoff + c0, pcount, kept_off, n_kept, hdr,
              scan_i);
}

// --------------------------------------------------------------- gather
// One warp per chunk writes its kept tokens (global index, position).
__global__ void __launch_bounds__(256) gather_write_kernel(
    const int32_t* seq_off, const int32_t* chunk_off, const uint8_t* keep, const int32_t* ckoff,
    const int32_t* kept_off, int32_t* kept_idx, int32_t* kept_pos, int B, int C, int force_bos,
    const int32_t* bad) {
    grid_dep_wait();
    grid_dep_launch();
    if (*bad) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cg = static_cast<int64_t>(blockIdx.x) * 8 + warp;
    if (cg >= chunk_off[B]) return;
    const int b = search_base(chunk_off, B, cg);
    const int64_t c = cg - chunk_off[b];
    const int64_t start = seq_off[b];
    const int64_t n = static_cast<int64_t>(seq_off[b + 1]) - start;
    const int64_t base = static_cast<int64_t>(kept_off[b]) + ckoff[cg];
    if (keep[cg]) {
        const int64_t a0 = c * C, a1 = min64(n, a0 + C);
        for (int64_t t = a0 + lane; t < a1; t += 32) {
            kept_idx[base + (t - a0)] = static_cast<int32_t>(start + t);
            kept_pos[base + (t - a0)] = static_cast<int32_t>(t);
        }
    } else if (c == 0 && force_bos && n > 0 && lane == 0) {
        kept_idx[base] = static_cast<int32_t>(start);
        kept_pos[base] = 0;
    }
}

}  // namespace

// ================================================================ launchers

cudaError_t launch_prep(const Plan& pl, const int32_t* seq_off, void* ws, int32_t* chunk_off_out,
                        cudaStream_t st, int64_t n_counters) {
    if (n_counters < 0) n_counters = (static_cast<int64_t>(pl.slabs_per_wave) + 1) * pl.B;
    return launch_k(prep_kernel, 1, kPrepThreads, 0, st, seq_off, pl.B, pl.Ntot, pl.C, pl.Tb,
        ws_ptr<int32_t>(ws, pl.o_tile_base),
        ws_ptr<int32_t>(ws, pl.o_chunk_off),
        ws_ptr<int32_t>(ws, pl.o_pblk_base), ws_ptr<int32_t>(ws, pl.o_slice_base), chunk_off_out,
        nullptr, ws_ptr<unsigned>(ws, pl.o_segcnt), n_counters, pl.kv_block_size,
        pl.kv_table_stride, pl.max_len, ws_ptr<WsHeader>(ws, 0));
}

cudaError_t launch_prep_check(const Plan& pl, const int32_t* seq_off, void* ws,
                              const int32_t* chunk_off_check, cudaStream_t st) {
    return launch_k(prep_kernel, 1, kPrepThreads, 0, st, seq_off, pl.B, pl.Ntot, pl.C, pl.Tb,
        ws_ptr<int32_t>(ws, pl.o_tile_base),
        ws_ptr<int32_t>(ws, pl.o_chunk_off),
        ws_ptr<int32_t>(ws, pl.o_pblk_base), ws_ptr<int32_t>(ws, pl.o_slice_base), nullptr,
        chunk_off_check, ws_ptr<unsigned>(ws, pl.o_segcnt),
        (static_cast<int64_t>(pl.slabs_per_wave) + 1) * pl.B, pl.kv_block_size, pl.kv_table_stride,
        pl.max_len, ws_ptr<WsHeader>(ws, 0));
}

cudaError_t launch_reduce(const Plan& pl, const int32_t* seq_off, void* ws, int nslab, int wave,
                          float* imp, cudaStream_t st) {
    if (pl.head_h > 0) return launch_reduce_head_pool(pl, seq_off, ws, nslab, wave, imp, st);
    const int tok = kReduceThreads / (pl.Rs / 8);
    const int nq = (tok + 31) / 32;
    const size_t smem = sizeof(float) * (static_cast<size_t>(nq) * nslab * pl.Rs +
                                         static_cast<size_t>(tok) * (pl.Rs + 1));
    auto kern = 8 % pl.G == 0 ? reduce_kernel<true> : reduce_kernel<false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const unsigned grid = static_cast<unsigned>(pl.tiles_max * (kTileTokens / tok));
    return launch_k(kern, grid, kReduceThreads, smem, st, ws_ptr<uint16_t>(ws, pl.o_logits),
                    ws_ptr<float>(ws, pl.o_lmax), ws_ptr<float>(ws, pl.o_lse), seq_off,
                    ws_ptr<int32_t>(ws, pl.o_tile_base), ws_ptr<float>(ws, pl.o_alog), imp, pl.B, pl.G, pl.L,
                    pl.R, pl.Rs, nslab, pl.Ntot, pl.tiles_max * kTileTokens, pl.tiles_max,
                    wave == 0 ? 1 : 0, wave == pl.waves - 1 ? 1 : 0, &ws_ptr<WsHeader>(ws, 0)->bad_input);
}

PoolArgs pool_args(const Plan& pl, const sp_params* p, const int32_t* seq_off, const float* imp,
                   float* tok, void* ws) {
    PoolArgs a;
    a.imp = imp;
    a.tok = tok;
    a.rpart = ws_ptr<float2>(ws, pl.o_rpart);
    a.csum = ws_ptr<float2>(ws, pl.o_csum);
    a.seq_off = seq_off;
    a.tile_base = ws_ptr<int32_t>(ws, pl.o_tile_base);
    a.chunk_off = ws_ptr<int32_t>(ws, pl.o_chunk_off);
    a.Ntot = pl.Ntot;
    a.B = pl.B;
    a.W = p->pool_w;
    a.C = pl.C;
    a.bf_n = p->boost_first_n;
    a.bl_n = p->boost_last_n;
    a.bf_mult = p->boost_first_mult;
    a.bl_mult = p->boost_last_mult;
    return a;
}

cudaError_t launch_pool_sums(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                             const float* imp, float* tok, void* ws, cudaStream_t st) {
    return launch_k(pool_sums_kernel, static_cast<unsigned>(pl.tiles_max), kPoolThreads, 0, st,
                    pool_args(pl, p, seq_off, imp, tok, ws), &ws_ptr<WsHeader>(ws, 0)->bad_input);
}

cudaError_t launch_pool(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                        const float* imp, float* tok, void* ws, cudaStream_t st) {
    const size_t smem = sizeof(float) * static_cast<size_t>(pl.Tb + 2 * (p->pool_w / 2));
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(pool_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_k(pool_kernel, static_cast<unsigned>(pl.pblk_max), 256, smem, st,
        imp, tok, ws_ptr<float2>(ws, pl.o_ppart), seq_off, ws_ptr<int32_t>(ws, pl.o_pblk_base),
        pl.B, p->pool_w, pl.Tb, &ws_ptr<WsHeader>(ws, 0)->bad_input);
}

cudaError_t launch_chunk(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                         const float* tok, float* chunk_score, void* ws, cudaStream_t st) {
    const size_t smem = sizeof(float) * static_cast<size_t>(pl.Tb);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_k(chunk_kernel, static_cast<unsigned>(pl.pblk_max), 256, smem, st,
        tok, ws_ptr<float2>(ws, pl.o_ppart), chunk_score, seq_off,
        ws_ptr<int32_t>(ws, pl.o_pblk_base), ws_ptr<int32_t>(ws, pl.o_chunk_off), pl.B, pl.C, pl.Tb,
        p->normalize, p->boost_first_mult, p->boost_first_n, p->boost_last_mult, p->boost_last_n,
        &ws_ptr<WsHeader>(ws, 0)->bad_input);
}

cudaError_t launch_select(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                          const int32_t* chunk_off, const float* chunk_score, uint8_t* keep,
                          void* ws, bool fuse_scan, int32_t* kept_off, int32_t* n_kept,
                          cudaStream_t st) {
    (void)seq_off;
    (void)fuse_scan;
    (void)kept_off;
    (void)n_kept;
    const int64_t max_nc = (pl.Ntot + pl.C - 1) / pl.C;
    (void)max_nc;
    const size_t smem = ((sizeof(SelectShared) + 15) & ~size_t(15)) + static_cast<size_t>(kMaxPromptChunks) * 5;
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(select_kernel, static_cast<unsigned>(pl.B), kSelThreads, smem, st,
        chunk_off, chunk_score, keep, ws_ptr<WsHeader>(ws, 0), p->mode, p->keep_p, p->mass,
        p->force_last_chunk);
}

cudaError_t launch_gather_scan(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                               const int32_t* chunk_off, const uint8_t* keep, void* ws,
                               int32_t* kept_off, int32_t* n_kept, cudaStream_t st) {
    return launch_k(gather_scan_kernel, static_cast<unsigned>(pl.B), kSelThreads, 0, st,
        seq_off, chunk_off, keep, ws_ptr<int32_t>(ws, pl.o_ckoff), ws_ptr<int32_t>(ws, pl.o_pcount),
        kept_off, n_kept, ws_ptr<WsHeader>(ws, 0), pl.B, pl.C, p->force_bos);
}

cudaError_t launch_gather_write(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                                const int32_t* chunk_off, const uint8_t* keep, int32_t* kept_idx,
                                int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept, void* ws,
                                cudaStream_t st) {
    (void)n_kept;
    const unsigned grid = static_cast<unsigned>((pl.chunks_max + 7) / 8);
    return launch_k(gather_write_kernel, grid, 256, 0, st, seq_off, chunk_off, keep,
                    ws_ptr<int32_t>(ws, pl.o_ckoff), kept_off, kept_idx, kept_pos, pl.B, pl.C,
                    p->force_bos, &ws_ptr<WsHeader>(ws, 0)->bad_input);
}

}  // namespace sp

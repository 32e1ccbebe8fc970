// Post-processing of the fused SpecPrefill scoring path, after the pool
// kernel has written the pooled scores (W-window mean, llama.cpp PR
// "Speculative prefill" §Approach item 3), their per-tile min / max and the
// per-chunk sums of boost * x and boost.
//
// The gather kernel runs one CTA per slice of kSliceChunks consecutive
// chunks of a prompt, the rank kernel one or kRankSplitMax CTAs per slice
// (each ranks its share of the slice's chunks), so a long prompt is spread
// over many SMs (the per-slice code is in sp_phases.cuh):
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
//           flags and the kept-token count of its part of the slice (chunk
//           0 counts its BOS token when it is not selected).
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

#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_phases.cuh"
#include "sp_select.cuh"

namespace sp {
namespace {

template <int SPLIT>
__global__ void __launch_bounds__(kRankThreads) rank_kernel(const PostArgs a) {
    // no early release: a dependent released early parks its CTAs on the
    // SMs its predecessor frees first; launched at this kernel's end it
    // spreads over every SM (with the same change in the logits, importance
    // and pool kernels: 2B workload 66.7 -> 64.1 us per call, 0.8B 39.4 ->
    // 35.2, long 257.8 -> 249.2)
    grid_dep_wait();
    const int64_t s = blockIdx.x / SPLIT;
    const int sub = static_cast<int>(blockIdx.x - s * SPLIT);
    extern __shared__ float cs_s[];  // the prompt's chunk scores
    __shared__ RankShared sh;
    if (a.B == 1) {  // rank_slice reads the flag after requesting its inputs
        const int64_t nc = (a.Ntot + a.C - 1) / a.C;
        const int64_t hi[3] = {a.Ntot, nc, (a.Ntot + kTileTokens - 1) / kTileTokens};
        const Located<3> loc = one_prompt<3>(static_cast<int32_t>((nc + kSliceChunks - 1) / kSliceChunks), hi);
        if (s >= loc.total) return;
        rank_slice<SPLIT>(a, s, sub, threadIdx.x, GroupBar{1, kRankThreads}, cs_s, sh, loc, &a.hdr->bad_input);
        return;
    }
    const int32_t* const aux[3] = {a.seq_off, a.chunk_off, a.tile_base};
    const int32_t bad_v = a.hdr->bad_input;
    const Located<3> loc = locate<3>(a.slice_base, aux, a.B, s);
    if (bad_v) return;
    if (s >= loc.total) return;
    rank_slice<SPLIT>(a, s, sub, threadIdx.x, GroupBar{1, kRankThreads}, cs_s, sh, loc, nullptr);
}

// One CTA per slice, plus one past the last slice for the totals.
__global__ void __launch_bounds__(kRankThreads) gather_kernel(const PostArgs a) {
    // no early release either: its successor is the next call's prep kernel
    // (2B workload 64.1 -> 63.5 us per call, 0.8B 35.3 -> 35.2)
    grid_dep_wait();
    __shared__ RankShared sh;
    const int64_t s = blockIdx.x;
    if (a.B == 1) {  // gather_slice reads the flag after requesting its inputs
        const int64_t nc = (a.Ntot + a.C - 1) / a.C;
        const int64_t hi[2] = {a.Ntot, nc};
        const Located<2> loc = one_prompt<2>(static_cast<int32_t>((nc + kSliceChunks - 1) / kSliceChunks), hi);
        if (s > loc.total) return;
        gather_slice(a, s, threadIdx.x, GroupBar{1, kRankThreads}, sh, loc, &a.hdr->bad_input);
        return;
    }
    const int32_t* const aux[2] = {a.seq_off, a.chunk_off};
    const int32_t bad_v = a.hdr->bad_input;
    const Located<2> loc = locate<2>(a.slice_base, aux, a.B, s);
    if (bad_v) return;
    if (s > loc.total) return;
    gather_slice(a, s, threadIdx.x, GroupBar{1, kRankThreads}, sh, loc, nullptr);
}

// Listing rule: the final kept count of prompt b from its count before the
// fill (the rank kernel's per-prompt sum): the fill up to eff_min, limited
// to the tokens the prompt has, then the cap.
__device__ __forceinline__ int64_t listing_final_count(const PostArgs& a, int b) {
    const int64_t n = static_cast<int64_t>(a.seq_off[b + 1]) - a.seq_off[b];
    const int64_t nc = static_cast<int64_t>(a.chunk_off[b + 1]) - a.chunk_off[b];
    if (nc == 0 || nc > kMaxPromptChunks) return 0;  // nothing kept (the latter reported by the rank)
    const int64_t k0 = __ldcg(a.lcount + b);
    const int64_t fill = min64(max64(0, listing_eff_min(n, a.min_tok) - k0), n - k0);
    const int64_t k = k0 + fill;
    return (a.max_keep > 0 && k > a.max_keep) ? a.max_keep : k;
}

// Listing rule gather, one CTA per slice of kSliceChunks chunks plus one
// for the totals. The prompt's kept list before the cap is: the tokens of
// its selected chunks and its forced tokens ("kept0"), plus the first
// `fill` of the remaining tokens ("spare") in token order. A kept0 token's
// position in that list is the number of kept0 tokens before it plus
// min(fill, spare tokens before it); a spare token is kept when fewer than
// `fill` spare tokens precede it. With the cap (count k > max_keep = M,
// step = k / M), position p goes to slot p / step when p % step == 0 and
// p / step < M - 1, and position k - 1 to slot M - 1; other positions are
// dropped. The counts before the slice come from the rank kernel's
// per-slice kept0 (scount) and spare (ucount) counts, those before each
// chunk from a scan over the slice's chunks, those before each token from
// warp ballots.
__global__ void __launch_bounds__(kRankThreads) listing_gather_kernel(const PostArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    __shared__ int64_t red[3][kRankWarps];
    __shared__ int64_t base_k[kSliceChunks], base_u[kSliceChunks];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t s = blockIdx.x;
    // A single prompt (B = 1) has seq_off = {0, Ntot} once the prep kernel
    // has accepted the input: its slice count follows from Ntot, and the
    // slice's counts, the prompt's count before the fill and the slice's
    // keep flags are requested before the flag is read.
    const bool one = a.B == 1;
    int64_t S;
    int64_t k0_one = 0;
    uint8_t f_one = 0;
    int64_t part[3] = {0, 0, 0};
    if (one) {
        const int64_t nc1 = (a.Ntot + a.C - 1) / a.C;
        S = (nc1 + kSliceChunks - 1) / kSliceChunks;
        if (s > S) return;
        if (s < S) {
            k0_one = __ldcg(a.lcount);
            if (warp == 0 && s * kSliceChunks + lane < nc1) f_one = __ldcg(a.keep + s * kSliceChunks + lane);
        }
        for (int64_t i = t; i < s * a.rank_split; i += kRankThreads) {
            part[1] += __ldcg(a.scount + i);
            part[2] += __ldcg(a.ucount + i);
        }
        if (a.hdr->bad_input) return;
    } else {
        if (a.hdr->bad_input) return;
        S = a.slice_base[a.B];
        if (s > S) return;
    }
    const int b = one ? 0 : (s == S ? a.B : search_base(a.slice_base, a.B, s));
    const int64_t sb = one ? 0 : (s == S ? S : a.slice_base[b]);
    // output offset of prompt b (final counts of all earlier prompts) and
    // the kept0 / spare tokens of the prompt's slices before this one
    if (!one) {
        for (int bb = t; bb < b; bb += kRankThreads) part[0] += listing_final_count(a, bb);
        for (int64_t i = sb * a.rank_split + t; i < s * a.rank_split; i += kRankThreads) {
            part[1] += __ldcg(a.scount + i);
            part[2] += __ldcg(a.ucount + i);
        }
    } else if (s == S && t == 0) {
        part[0] = listing_final_count(a, 0);  // the totals CTA: the prompt's final count
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        for (int o = 16; o > 0; o >>= 1) part[j] += __shfl_xor_sync(0xffffffffu, part[j], o);
        if (lane == 0) red[j][warp] = part[j];
    }
    __syncthreads();
    int64_t P = 0, kb0 = 0, ub0 = 0;
    for (int w = 0; w < kRankWarps; ++w) {
        P += red[0][w];
        kb0 += red[1][w];
        ub0 += red[2][w];
    }
    if (s == S) {
        if (t == 0) {
            for (int bb = a.B - 1; !one && bb >= 0 && a.slice_base[bb] == S; --bb)
                a.kept_off[bb] = static_cast<int32_t>(P);
            a.kept_off[a.B] = static_cast<int32_t>(P);
            *a.n_kept = static_cast<int32_t>(P);
        }
        return;
    }
    if (t == 0 && s == sb) {
        // first slice of prompt b: its offset, and that of empty prompts before it
        a.kept_off[b] = static_cast<int32_t>(P);
        for (int bb = b - 1; bb >= 0 && a.slice_base[bb] == s; --bb) a.kept_off[bb] = static_cast<int32_t>(P);
    }
    const int64_t start = one ? 0 : a.seq_off[b];
    const int64_t n = one ? a.Ntot : static_cast<int64_t>(a.seq_off[b + 1]) - start;
    const int64_t coff = one ? 0 : a.chunk_off[b];
    const int64_t nc = one ? (a.Ntot + a.C - 1) / a.C : static_cast<int64_t>(a.chunk_off[b + 1]) - coff;
    if (nc > kMaxPromptChunks) return;  // reported by the rank kernel; nothing kept
    const int64_t k0 = one ? k0_one : __ldcg(a.lcount + b);
    const int64_t fill = min64(max64(0, listing_eff_min(n, a.min_tok) - k0), n - k0);
    const int64_t k = k0 + fill;
    const int64_t M = (a.max_keep > 0 && k > a.max_keep) ? a.max_keep : 0;
    const int64_t step = M > 0 ? k / M : 1;
    const int64_t c_lo = (s - sb) * kSliceChunks;
    // exclusive scans of the slice's per-chunk kept0 / spare counts (lane = chunk)
    if (warp == 0) {
        const int64_t c = c_lo + lane;
        int64_t ck = 0, cu = 0;
        if (c < nc) {
            const int64_t a0 = c * a.C, a1 = a0 + chunk_tokens(n, a.C, c);
            if ((one ? f_one : __ldcg(a.keep + coff + c)) & 1) {
                ck = a1 - a0;
            } else {
                ck = listing_forced_in(a0, a1, n);
                cu = a1 - a0 - ck;
            }
        }
        int64_t ik = ck, iu = cu;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t vk = __shfl_up_sync(0xffffffffu, ik, o);
            const int64_t vu = __shfl_up_sync(0xffffffffu, iu, o);
            if (lane >= o) {
                ik += vk;
                iu += vu;
            }
        }
        base_k[lane] = kb0 + ik - ck;
        base_u[lane] = ub0 + iu - cu;
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int q = warp; q < kSliceChunks; q += kRankWarps) {
        const int64_t c = c_lo + q;
        if (c >= nc) break;
        const int64_t a0 = c * a.C, a1 = a0 + chunk_tokens(n, a.C, c);
        const bool sel = (__ldcg(a.keep + coff + c) & 1) != 0;
        int64_t kb = base_k[q], ub = base_u[q];
        for (int64_t g0 = a0; g0 < a1; g0 += 32) {
            const int64_t tt = g0 + lane;
            const bool in = tt < a1;
            const bool kept0 = in && (sel || listing_forced(tt, n));
            const bool spare = in && !kept0;
            const unsigned km = __ballot_sync(0xffffffffu, kept0);
            const unsigned um = __ballot_sync(0xffffffffu, spare);
            const int64_t kbt = kb + __popc(km & lt), ubt = ub + __popc(um & lt);
            int64_t p = -1;
            if (kept0) p = kbt + min64(fill, ubt);
            else if (spare && ubt < fill) p = kbt + ubt;
            if (p >= 0) {
                int64_t slot = p;
                if (M > 0) {
                    if (p == k - 1) slot = M - 1;
                    else if (p % step == 0 && p / step < M - 1) slot = p / step;
                    else slot = -1;
                }
                if (slot >= 0) {
                    a.kept_idx[P + slot] = static_cast<int32_t>(start + tt);
                    a.kept_pos[P + slot] = static_cast<int32_t>(tt);
                }
            }
            kb += __popc(km);
            ub += __popc(um);
        }
    }
}

}  // namespace

PostArgs post_args(const Plan& pl, const sp_params* p, const int32_t* seq_off, float* chunk_score,
                   uint8_t* keep, int32_t* kept_idx, int32_t* kept_pos, int32_t* kept_off,
                   int32_t* n_kept, void* ws) {
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
    a.lcount = ws_ptr<int32_t>(ws, pl.o_lcount);
    a.ucount = ws_ptr<int32_t>(ws, pl.o_ucount);
    a.hdr = ws_ptr<WsHeader>(ws, 0);
    a.B = pl.B;
    a.Ntot = pl.Ntot;
    a.C = pl.C;
    a.mode = p->mode;
    a.normalize = p->normalize;
    a.force_bos = p->force_bos;
    a.force_last = p->force_last_chunk;
    a.keep_p = p->keep_p;
    a.mass = p->mass;
    a.rule = p->rule;
    a.min_tok = p->min_tok;
    a.max_keep = p->max_keep;
    a.rank_split = 1;
    return a;
}

cudaError_t launch_post(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                        float* chunk_score, uint8_t* keep, int32_t* kept_idx, int32_t* kept_pos,
                        int32_t* kept_off, int32_t* n_kept, void* ws, cudaStream_t st) {
    PostArgs a = post_args(pl, p, seq_off, chunk_score, keep, kept_idx, kept_pos, kept_off, n_kept, ws);
    // Few slices: kRankSplitMax CTAs per slice, one warp per chunk, so that
    // the ranking scans run on more SMs (2B workload 63.3 -> 62.5 us per
    // call, 0.8B 34.8 -> 34.4); with more slices than the SMs hold that way,
    // every CTA rebuilding all chunk scores costs more than it saves (long
    // workload 243.7 -> 251.0 with four CTAs per slice, 239.0 -> 240.4 with
    // two), so one CTA ranks the whole slice.
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    a.rank_split = pl.slices_max * kRankSplitMax <= sms ? kRankSplitMax : 1;
    auto kern = a.rank_split == 1 ? rank_kernel<1> : rank_kernel<kRankSplitMax>;
    // shared memory for the largest prompt's chunk scores
    const int64_t maxnc = pl.chunks_max < kMaxPromptChunks ? pl.chunks_max : kMaxPromptChunks;
    const size_t smem = static_cast<size_t>(maxnc) * sizeof(float);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const cudaError_t e =
        launch_k(kern, static_cast<unsigned>(pl.slices_max * a.rank_split), kRankThreads, smem, st, a);
    if (e != cudaSuccess) return e;
    if (p->rule == SP_RULE_LISTING)
        return launch_k(listing_gather_kernel, static_cast<unsigned>(pl.slices_max + 1), kRankThreads, 0, st, a);
    return launch_k(gather_kernel, static_cast<unsigned>(pl.slices_max + 1), kRankThreads, 0, st, a);
}

}  // namespace sp

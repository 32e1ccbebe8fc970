// Post-processing of the fused SpecPrefill scoring path, after the pool
// kernel has written the pooled scores (W-window mean, llama.cpp PR
// "Speculative prefill" §Approach item 3), their per-tile min / max and the
// per-chunk sums of boost * x and boost.
//
// Both kernels run one CTA per slice of kSliceChunks consecutive chunks of a
// prompt, so a long prompt is spread over many SMs (the per-slice code is in
// sp_phases.cuh, shared with the persistent fused kernel):
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

#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_phases.cuh"

namespace sp {
namespace {

__global__ void __launch_bounds__(kRankThreads) rank_kernel(const PostArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    if (a.hdr->bad_input) return;
    const int64_t s = blockIdx.x;
    if (s >= a.slice_base[a.B]) return;
    extern __shared__ float cs_s[];  // the prompt's chunk scores
    __shared__ RankShared sh;
    rank_slice(a, s, threadIdx.x, GroupBar{1, kRankThreads}, cs_s, sh);
}

// One CTA per slice, plus one past the last slice for the totals.
__global__ void __launch_bounds__(kRankThreads) gather_kernel(const PostArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    if (a.hdr->bad_input) return;
    __shared__ RankShared sh;
    const int64_t S = a.slice_base[a.B];
    const int64_t s = blockIdx.x;
    if (s > S) return;
    gather_slice(a, s, S, threadIdx.x, GroupBar{1, kRankThreads}, sh);
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
    a.hdr = ws_ptr<WsHeader>(ws, 0);
    a.B = pl.B;
    a.C = pl.C;
    a.mode = p->mode;
    a.normalize = p->normalize;
    a.force_bos = p->force_bos;
    a.force_last = p->force_last_chunk;
    a.keep_p = p->keep_p;
    a.mass = p->mass;
    return a;
}

cudaError_t launch_post(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                        float* chunk_score, uint8_t* keep, int32_t* kept_idx, int32_t* kept_pos,
                        int32_t* kept_off, int32_t* n_kept, void* ws, cudaStream_t st) {
    const PostArgs a = post_args(pl, p, seq_off, chunk_score, keep, kept_idx, kept_pos, kept_off, n_kept, ws);
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

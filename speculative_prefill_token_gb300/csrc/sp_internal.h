// Internal host/device declarations of the SpecPrefill library: the launch
// plan derived from a shape, the workspace layout, and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "specprefill.h"

namespace sp {

constexpr int kTileTokens = 128;   // tokens per logits tile (tensor-core M)
constexpr int kMaxRows = 64;       // max query rows per slab (L * G)
constexpr int kPostBlockTarget = 1024;
constexpr int kMaxSeqs = 65536;
constexpr int kMaxKvLayers = 64;    // per-layer key pools (one tensor map each, kernel parameters)
constexpr int kMaxChunk = 8192;
constexpr int kMaxPool = 8191;
constexpr int kMaxPromptChunks = 16384;  // per-prompt chunk count the in-CTA selection handles
constexpr int kSliceChunks = 32;         // chunks per CTA of the fused gather kernels
constexpr int kRankSplitMax = 4;        // rank CTAs per slice at most (each ranks kSliceChunks / split chunks)
constexpr int64_t kDefaultSpin = int64_t(1) << 22;  // ~4 s of polls with a 1 us suspend hint

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
    int32_t status;        // sticky device status (sp_status), written by kernels on failure
    int32_t bad_input;     // set by the prep kernel of the current call when seq_off is invalid
    uint32_t ticket;       // last-block-done counter of the gather scan (zeroed by prep)
    int32_t pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header size");

struct Plan {
    // shape
    int B, Ly, Hq, Hk, G, d, L, R, Rs, Nmma, Nacc;  // Rs = 32 or 64 (row stride of the scratch)
    int64_t Ntot;
    int slabs;
    int64_t tiles_max;    // >= sum_b ceil(n_b / 128)
    int64_t rec_slots;    // softmax records: (max CTAs + segments per wave) * 2 warpgroups
    int64_t chunks_max;   // >= sum_b ceil(n_b / C)
    int C, W;
    int64_t Tb;           // tokens per post-processing block (multiple of C)
    int64_t pblk_max;     // >= sum_b ceil(n_b / Tb)
    int64_t slices_max;   // >= sum_b ceil(ceil(n_b / C) / kSliceChunks)
    int sort_cap;         // power of two >= max chunks of one prompt
    int slabs_per_wave, waves;
    float scale2;         // logit scale * log2(e)
    int64_t spin;         // bounded-wait poll limit
    int max_len;          // longest prompt the caller allows (0 = no bound)
    int head_h;           // per-head pooling: half window (0 = pool the per-token importance)
    int kv_block_size, kv_table_stride;  // block-paged key source (checked by the prep kernel)
    // workspace offsets (bytes)
    size_t o_tile_base, o_chunk_off, o_pblk_base, o_slice_base, o_scount, o_segcnt, o_logits, o_lmax, o_part, o_lse, o_alog, o_imp, o_tok,
        o_rpart, o_csum,
        o_ppart, o_cscore, o_ckeep, o_ckoff, o_pcount, o_lcount, o_ucount, o_kept_off, o_nkept, total;
};

int make_plan(const sp_shape* s, const sp_params* p, Plan* plan);

// ------------------------------------------------------------ launchers
// Each returns cudaSuccess or the launch error.

// Per-call offsets and checks; also zeroes the per-segment record counters
// and the per-prompt kept counts of the listing rule (one range of
// n_counters words; < 0 selects the plan's own count).
cudaError_t launch_prep(const Plan& pl, const int32_t* seq_off, void* ws, int32_t* chunk_off_out,
                        cudaStream_t st, int64_t n_counters = -1);

// Logits of the slabs [slab0, slab0 + nslab) into the workspace scratch
// (one 128-row slot per tile), plus softmax records per (CTA, segment,
// warpgroup). Tensor-core (tcgen05 + TMA) kernel on `grid` CTAs.
int logits_tc_grid(const Plan& pl, int nslab);
// Keys held per layer by a draft engine: one pool per layer, addressed by
// the packed token index, or (block_table != nullptr) by blocks of
// block_size tokens through a per-prompt table of physical block ids.
struct KvSrc {
    const uint16_t* layer_k[kMaxKvLayers];
    const int32_t* block_table;  // [B][table_stride], device
    int block_size, table_stride;
    int64_t pool_tokens;         // token rows in each layer's pool
};
// With kv != nullptr the keys come from kv (k is unused).
cudaError_t launch_logits_tc(const Plan& pl, const sp_shape* s, const int32_t* seq_off,
                             const uint16_t* q, const uint16_t* k, void* ws, int slab0, int nslab,
                             int grid, cudaStream_t st, const KvSrc* kv = nullptr);


// Softmax, max over heads/layers of the wave; the last wave writes imp.
// With per-head pooling (pl.head_h > 0) every row is pooled before the max
// (sp_head_pool.cu).
cudaError_t launch_reduce(const Plan& pl, const int32_t* seq_off, void* ws, int nslab, int wave,
                          float* imp, cudaStream_t st);
cudaError_t launch_reduce_head_pool(const Plan& pl, const int32_t* seq_off, void* ws, int nslab,
                                    int wave, float* imp, cudaStream_t st);

// The selection parameters of the steps after the importance: with
// per-head pooling the pool has already been applied (width 1 afterwards).
inline sp_params post_params(const sp_params* p) {
    sp_params q = *p;
    if (q.pool_at == SP_POOL_HEAD) q.pool_w = 1;
    return q;
}

// Fused-path pooling: pooled scores, per-tile min / max and per-chunk sums
// (requires fused_post_ok: the pool halo fits and chunks never straddle a
// 128-token tile).
inline bool fused_post_ok(const sp_params* p) {
    return p->pool_w / 2 <= 64 && 128 % p->chunk == 0;
}
cudaError_t launch_pool_sums(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                             const float* imp, float* tok, void* ws, cudaStream_t st);

cudaError_t launch_pool(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                        const float* imp, float* tok, void* ws, cudaStream_t st);

cudaError_t launch_chunk(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                         const float* tok, float* chunk_score, void* ws, cudaStream_t st);

// CUDA-core cross-check of the logits kernel, same outputs; returns its
// grid (one work item per CTA) through *grid.
cudaError_t launch_logits_simt(const Plan& pl, const sp_shape* s, const int32_t* seq_off,
                               const uint16_t* q, const uint16_t* k, void* ws, int slab0, int nslab,
                               int* grid, cudaStream_t st);

cudaError_t launch_prep_check(const Plan& pl, const int32_t* seq_off, void* ws,
                              const int32_t* chunk_off_check, cudaStream_t st);

// Selection; when `fuse_scan` is set it also writes the per-chunk kept
// offsets, and the last prompt to finish writes kept_off / n_kept.
cudaError_t launch_select(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                          const int32_t* chunk_off, const float* chunk_score, uint8_t* keep,
                          void* ws, bool fuse_scan, int32_t* kept_off, int32_t* n_kept,
                          cudaStream_t st);

cudaError_t launch_gather_scan(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                               const int32_t* chunk_off, const uint8_t* keep, void* ws,
                               int32_t* kept_off, int32_t* n_kept, cudaStream_t st);

cudaError_t launch_gather_write(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                                const int32_t* chunk_off, const uint8_t* keep, int32_t* kept_idx,
                                int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept, void* ws,
                                cudaStream_t st);

// Fused post-processing after launch_pool_sums: the rank kernel (chunk
// scores, selection, force-last, kept tokens per 32-chunk slice) and the
// gather kernel (kept lists, per-prompt offsets, total), one CTA per slice.
cudaError_t launch_post(const Plan& pl, const sp_params* p, const int32_t* seq_off,
                        float* chunk_score, uint8_t* keep, int32_t* kept_idx, int32_t* kept_pos,
                        int32_t* kept_off, int32_t* n_kept, void* ws, cudaStream_t st);

// Sparse-prefill consumer gathers (sp_rows.cu): kept rows of a token-major
// bf16 cache tensor, and kept token ids.
cudaError_t launch_gather_rows(const sp_shape* s, const int32_t* kept_idx, const int32_t* n_kept,
                               const uint16_t* src, uint16_t* dst, int64_t dst_rows,
                               cudaStream_t st);
cudaError_t launch_merge_windows(int64_t n, int window, int stride, const float* imp_windows,
                                 float* out, cudaStream_t st);
cudaError_t launch_gather_tokens(const int32_t* ids, const int32_t* kept_idx, const int32_t* n_kept,
                                 int32_t* out, int64_t ntot, cudaStream_t st);

// Launch with programmatic stream serialisation: the kernel may be
// scheduled while its predecessor in the stream is still running and waits
// for it in grid_dep_wait() (every kernel of this library does so before
// touching global memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

template <typename T>
inline T* ws_ptr(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace sp

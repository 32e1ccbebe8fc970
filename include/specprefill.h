/*
 * specprefill.h — C ABI of the SpecPrefill token-importance and
 * chunk-selection path, hand-written CUDA for sm_103a (GB300).
 *
 * The path (pages: "SpecPrefill — Implementation Guide" of the
 * sliding-specprefill project, versions v2 and v3.1, and the llama.cpp pull
 * request "Speculative prefill"):
 *
 *   logits    s = scale * <q, k> for every lookahead query vector q of every
 *             attention layer and query head, against the prompt's cached
 *             keys k (GQA: query head h reads KV head h / (Hq/Hk))
 *   softmax   over the prompt's keys                    (guide §How It Works /
 *                                                        Attention Capture)
 *   importance  max over heads, max over layers, mean over lookahead steps
 *                                                       (guide §How It Works /
 *                                                        Token Importance)
 *   pool      centred average over W tokens (W = 13)    (PR §Approach item 3)
 *   normalise min-max to [0, 1] (optional)              (guide v3.1 item 5)
 *   boost     first 64 tokens x1.5, last 128 x1.3      (guide v3 item 2)
 *   chunks    mean score of 32-token chunks             (guide §Chunk Selection)
 *   select    top k = max(1, ceil(nc * p)) chunks, or the shortest ranked
 *             prefix holding `mass` of the total score  (guide v3 item 1)
 *   force     BOS and each prompt's final chunk         (PR §Approach item 4)
 *   gather    kept token indices + original position IDs (guide §How It
 *                                                        Works / Sparse Prefill)
 *
 * Conventions for every entry point
 * - Pointers marked (device) are device memory owned by the caller; the
 *   library never allocates, frees or retains them, and keeps no state
 *   between calls. Pointers marked (host) are host memory read during the
 *   call.
 * - Work is enqueued on `stream` and runs asynchronously; no entry point
 *   synchronises except sp_get_device_status.
 * - Return value: SP_OK, or an sp_status code for an argument the host can
 *   check (nothing is enqueued then) or a launch error. Faults the device
 *   detects itself (a bounded wait that gave up) set a sticky status word in
 *   the workspace, read with sp_get_device_status.
 * - Ranking ties break by ascending chunk index; the fixed mode keeps
 *   exactly k ranked chunks.
 * - Prompts are packed along the token axis: prompt b owns global tokens
 *   [seq_off[b], seq_off[b+1]). Chunks never cross prompts; prompt b owns
 *   chunks [chunk_off[b], chunk_off[b+1]), chunk_off[b+1]-chunk_off[b] =
 *   ceil(n_b / chunk).
 */
#ifndef SPECPREFILL_H
#define SPECPREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t / cudaEvent_t. */
typedef struct CUstream_st* sp_stream_t;
typedef struct CUevent_st* sp_event_t;

typedef enum sp_status {
    SP_OK = 0,
    SP_ERR_INVALID_ARG = 1,   /* null pointer, inconsistent shape, parameter out of range */
    SP_ERR_UNSUPPORTED = 2,   /* head_dim not in {64,128,256}, L*G > 64, misaligned strides */
    SP_ERR_WORKSPACE = 3,     /* workspace null, misaligned (256 B) or smaller than required */
    SP_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    SP_ERR_TIMEOUT = 5,       /* (device status) a bounded device wait gave up */
    SP_ERR_DEVICE = 6         /* (device status) the kernel found an inconsistent input */
} sp_status;

enum { SP_MODE_FIXED = 0, SP_MODE_MASS = 1 };

/* Selection rule.
 * SP_RULE_EXACT: exactly k chunks in fixed mode (ties broken by ascending
 *   chunk index), token 0 and the final chunk forced (force_bos,
 *   force_last_chunk); the SpecPrefill scoring contract.
 * SP_RULE_LISTING: the rule of the pages' own tool ("SpecPrefill —
 *   Implementation Guide", v2 listing `select_chunks` and the cap in `main`):
 *   k = max(1, ceil(nc * p)) with the product rounded to float32, every
 *   chunk scoring at least the k-th largest score kept (ties can keep more
 *   than k), tokens {0, 1, 2, 3, n-2, n-1} forced (the last two when
 *   n > 4; force_bos and force_last_chunk are ignored), then a fill of the
 *   smallest unselected tokens up to eff_min = min(min_tok, max(4, n / 10))
 *   tokens, everything kept when p >= 1 (fixed mode) or n <= eff_min, and
 *   finally, when max_keep > 0 and more than max_keep tokens are kept, every
 *   step-th kept token (step = count / max_keep) up to max_keep of them with
 *   the last one replaced by the prompt's last kept token. Mass mode keeps
 *   its ranking prefix and then applies the forced tokens, the fill and the
 *   cap. Only sp_specprefill_score and sp_select_from_importance take this
 *   rule, and only with pool_w / 2 <= 64 and chunk dividing 128
 *   (SP_ERR_UNSUPPORTED otherwise). */
enum { SP_RULE_EXACT = 0, SP_RULE_LISTING = 1 };

/* Where the W-wide average pool applies (llama.cpp PR "Speculative
 * prefill", §Approach item 3, lists the smoothing together with the max over
 * heads and layers without fixing the order).
 * SP_POOL_TOKEN: on the per-token importance, after the mean over the
 *   lookahead steps (the scoring contract).
 * SP_POOL_HEAD: on every attention row (layer, step, query head) before the
 *   max over heads and layers; the later pooling step is then the identity
 *   (sp_pool_chunk and the fused call treat pool_w as 1 after it). Requires
 *   pool_w / 2 <= 64 (SP_ERR_UNSUPPORTED otherwise). */
enum { SP_POOL_TOKEN = 0, SP_POOL_HEAD = 1 };

/* Shapes and strides. Strides are in elements; the head_dim axis is
 * contiguous (stride 1).
 * K: bf16 keys of layer l, global token t, KV head g at
 *    k[l*k_stride_layer + t*k_stride_token + g*k_stride_head + j]
 *    (a token-major KV cache, e.g. [Ly][Ntot][Hk][d] contiguous).
 * Q: bf16 lookahead queries of prompt b, layer l, step s, query head h at
 *    q[b*q_stride_seq + l*q_stride_layer + s*q_stride_step + h*q_stride_head + j]
 *    (e.g. [B][Ly][L][Hq][d] contiguous).
 * Every stride times 2 bytes must be a multiple of 16 and both base
 * pointers 16-byte aligned (tensor-memory-accelerator tiles). */
typedef struct sp_shape {
    int32_t n_seqs;          /* B >= 1 prompts */
    int32_t n_layers;        /* Ly >= 1 attention layers */
    int32_t n_q_heads;       /* Hq >= 1 */
    int32_t n_kv_heads;      /* Hk >= 1, Hq % Hk == 0, G = Hq / Hk */
    int32_t head_dim;        /* d in {64, 128, 256} */
    int32_t n_lookahead;     /* L >= 1 query vectors per layer and head; L*G <= 64 */
    int32_t n_tokens_total;  /* Ntot = seq_off[B] >= 1 */
    int32_t max_seq_len;     /* 0 (no bound), or the longest prompt the caller
                                allows: a prompt with more tokens makes the
                                call's device status SP_ERR_DEVICE (checked on
                                the device with seq_off); < 0 is invalid */
    int64_t k_stride_layer, k_stride_token, k_stride_head;
    int64_t q_stride_seq, q_stride_layer, q_stride_step, q_stride_head;
} sp_shape;

typedef struct sp_params {
    int32_t pool_w;            /* odd, >= 1 (13); 1 = no smoothing */
    int32_t chunk;             /* C >= 1 (32) */
    int32_t mode;              /* SP_MODE_FIXED or SP_MODE_MASS */
    float keep_p;              /* fixed mode, in (0, 1] (0.30) */
    float mass;                /* mass mode, in (0, 1] (0.85) */
    int32_t normalize;         /* 1: min-max normalise each prompt's pooled scores */
    float boost_first_mult;    /* > 0 (1.5); 1 = off */
    int32_t boost_first_n;     /* >= 0 (64) */
    float boost_last_mult;     /* > 0 (1.3); 1 = off */
    int32_t boost_last_n;      /* >= 0 (128) */
    int32_t force_bos;         /* 1: token 0 of every prompt is kept */
    int32_t force_last_chunk;  /* 1: every prompt's final chunk is kept */
    float scale;               /* logit scale; 0 selects 1/sqrt(head_dim) */
    int32_t spin_limit;        /* polls before a device wait gives up; <= 0 selects the default */
    int32_t rule;              /* SP_RULE_EXACT (0) or SP_RULE_LISTING */
    int32_t min_tok;           /* SP_RULE_LISTING: >= 0 (128), bound of eff_min */
    int32_t max_keep;          /* SP_RULE_LISTING: >= 0 (2000 in the pages' tool); 0 = no cap */
    int32_t pool_at;           /* SP_POOL_TOKEN (0) or SP_POOL_HEAD */
    int32_t wave_mib;          /* >= 0; 0 selects the default (2048). The logits
                                  of all slabs are kept in the workspace between
                                  the two passes of the softmax; when they need
                                  more than this many MiB the slabs are scored in
                                  waves that each fit it (smaller workspace, one
                                  more pair of kernels per wave) */
} sp_params;

/* Optional profiling hook: when non-null, `logits_start`/`logits_stop` are
 * recorded on `stream` immediately around the logits kernel(s). */
typedef struct sp_profile {
    sp_event_t logits_start;
    sp_event_t logits_stop;
} sp_profile;

/* Number of kernels one sp_specprefill_score call with this shape and these
 * parameters launches on its stream (all of them this library's own), so a
 * caller can account for the launches it issues. */
int sp_kernels_per_call(const sp_shape* shape, const sp_params* params, int32_t* n_kernels);

/* Upper bound on the number of chunks of a packed batch:
 * floor(Ntot / chunk) + B. Chunk arrays must hold this many entries. */
int sp_max_chunks(const sp_shape* shape, const sp_params* params, int64_t* n_chunks);

/* Bytes of device workspace the entry points below need for this shape on
 * the current device (writes *bytes). */
int sp_workspace_size(const sp_shape* shape, const sp_params* params, size_t* bytes);

/* Zero the workspace's status word. Call once on a new workspace (or use
 * zero-filled memory) before the first call that uses it. */
int sp_workspace_init(void* ws, size_t ws_bytes, sp_stream_t stream);

/* Token importance (logits, softmax, max over heads and layers, mean over
 * steps): imp[t] for every global token t (device, Ntot floats).
 * Defined by "SpecPrefill — Implementation Guide", §How It Works / Attention
 * Capture (one post-softmax attention row per head and lookahead step over
 * the prompt's keys) and §How It Works / Token Importance (max over heads,
 * then max over layers, then the mean over the lookahead steps); the draft's
 * L lookahead queries and full-attention layers are those of llama.cpp PR
 * "Speculative prefill", §Approach items 1-2.
 * seq_off (device, B+1 int32, non-decreasing from 0 to Ntot), q and k
 * (device, bf16 bits) as described at sp_shape. */
int sp_attn_importance(const sp_shape* shape, const sp_params* params,
                       const int32_t* seq_off, const uint16_t* q, const uint16_t* k,
                       float* imp, void* ws, size_t ws_bytes, sp_stream_t stream);

/* Same contract as sp_attn_importance, but the logits come from a CUDA-core
 * (FP32 FMA) kernel instead of the tensor-core one. It exists as an
 * independent cross-check of the tensor-core kernel in the GPU tests. */
int sp_attn_importance_simt(const sp_shape* shape, const sp_params* params,
                            const int32_t* seq_off, const uint16_t* q, const uint16_t* k,
                            float* imp, void* ws, size_t ws_bytes, sp_stream_t stream);

/* Smoothing and chunk scores from imp (device, Ntot floats).
 * Defined by llama.cpp PR "Speculative prefill", §Approach item 3 (the
 * W-wide average pool), "SpecPrefill — Implementation Guide" v3.1, §v3.1
 * Optimizations item 5 (min-max normalisation), v3 §v3 Improvements item 2
 * (structural boost of the first and last tokens) and §Chunk Selection (a
 * chunk's score is the mean of its tokens' scores).
 * tok_score (device, Ntot floats, nullable): pooled score before
 * normalisation and boost. chunk_score (device, sp_max_chunks floats): the
 * final chunk scores. chunk_off (device, B+1 int32): written. */
int sp_pool_chunk(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                  const float* imp, float* tok_score, float* chunk_score, int32_t* chunk_off,
                  void* ws, size_t ws_bytes, sp_stream_t stream);

/* Allocation-free variant of sp_pool_chunk (the pages have no counterpart;
 * this entry point exists for callers that cannot allocate device memory:
 * code running under a memory pool that owns all device memory and forbids
 * allocations after start-up, plugins whose host runtime gives them no
 * allocator, or loops that must not risk the device synchronisation a
 * cudaMalloc/cudaFree can cause). Same results as sp_pool_chunk, without a
 * workspace: its scratch lives in a fixed 1 MiB array inside the library on
 * every GPU that loads it, kept until the process exits. It calls no
 * allocation routine.
 * - tok_score, chunk_score (sp_max_chunks floats) and chunk_off (B+1) are
 *   required device outputs.
 * - status_out (device, one int32, nullable) receives this call's device
 *   status in stream order: SP_OK, or SP_ERR_DEVICE when seq_off is invalid.
 * - Batches whose scratch does not fit return SP_ERR_UNSUPPORTED before
 *   anything is enqueued. The scratch is a 256-byte header, four offset
 *   tables of 4*(B+1) bytes each (each rounded up to 256 bytes) and 8 bytes
 *   per pooling block of floor(1024 / chunk) * chunk tokens (one block per
 *   1024 tokens at chunk 32, plus one per prompt); it depends on B, Ntot and
 *   chunk only. At chunk 32 that admits, for example, 16,000 prompts of 1K
 *   tokens or one prompt of 100M tokens.
 * - Each call looks up the array's device address in the calling thread's
 *   current CUDA context (a new context after cudaDeviceReset, or another
 *   context on the same GPU, has its own copy of the array) unless the
 *   stream is being captured; a call made during stream capture reuses the
 *   address the last uncaptured call on that context found, so make one
 *   uncaptured call per context first.
 * - All calls on one GPU share the array and each leaves its contents
 *   behind: calls that overlap on the GPU (unordered streams or threads)
 *   race, so order them on one stream. */
int sp_pool_chunk_noalloc(const sp_shape* shape, const sp_params* params,
                          const int32_t* seq_off, const float* imp, float* tok_score,
                          float* chunk_score, int32_t* chunk_off, int32_t* status_out,
                          sp_stream_t stream);

/* Chunk selection per prompt, defined by "SpecPrefill — Implementation
 * Guide", §Chunk Selection (the top k = max(1, ceil(nc * p)) chunks by
 * score), v3 §v3 Improvements item 1 (cumulative attention mass: the
 * shortest ranked prefix holding `mass` of the total) and llama.cpp PR
 * "Speculative prefill", §Approach item 4 (BOS and the final chunk are always
 * kept). chunk_keep (device, one byte per chunk):
 * bit 0 = chosen by the ranking, bit 1 = forced final chunk.
 * SP_RULE_LISTING is not a chunk-level rule: SP_ERR_UNSUPPORTED (likewise
 * for sp_gather_kept). */
int sp_select(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
              const int32_t* chunk_off, const float* chunk_score, uint8_t* chunk_keep,
              void* ws, size_t ws_bytes, sp_stream_t stream);

/* Stream compaction of kept tokens, defined by "SpecPrefill —
 * Implementation Guide", §How It Works / Sparse Prefill (the target
 * prefills only the kept tokens, each at its original position ID). For
 * prompt b, its kept tokens (those
 * in a chunk with chunk_keep != 0, plus token 0 when force_bos) in
 * increasing order occupy [kept_off[b], kept_off[b+1]) of kept_idx (global
 * token index) and kept_pos (position within the prompt, i.e. the original
 * position ID). kept_idx/kept_pos: device, capacity Ntot int32 each;
 * kept_off: device, B+1 int32; n_kept: device, 1 int32 (= kept_off[B]). */
int sp_gather_kept(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                   const int32_t* chunk_off, const uint8_t* chunk_keep, int32_t* kept_idx,
                   int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept, void* ws,
                   size_t ws_bytes, sp_stream_t stream);

/* Sparse-prefill consumer: the rows of the kept tokens of a token-major
 * cache tensor ("SpecPrefill — Implementation Guide", §How It Works / Sparse
 * Prefill: the target prefills only the kept tokens, each at its original
 * position), so that keys or values built from the draft can be handed to
 * the target compactly.
 * - src (device, bf16 bits): [Ly][Ntot][Hk][d] with the k_stride_* strides
 *   of `shape` (d contiguous); only Ly, Ntot, Hk, d and those strides of
 *   `shape` are used.
 * - kept_idx (device, int32): packed token indices, e.g. from
 *   sp_specprefill_score; n_kept (device, one int32): how many of them to
 *   gather. Both are read on the device, so no host synchronisation is
 *   needed between the selection and this call.
 * - dst (device, bf16 bits): [Ly][dst_rows][Hk][d], dense; row i of layer l
 *   receives src[l][kept_idx[i]]. dst_rows must be at least Ntot (the
 *   largest possible kept count); rows past n_kept are left untouched.
 * - An index outside [0, Ntot) gives a zero row; n_kept is clamped to
 *   [0, Ntot].
 * Returns SP_ERR_INVALID_ARG for a bad shape, a null pointer, a pointer that
 * is not 16-byte aligned or dst_rows < Ntot. */
int sp_gather_rows(const sp_shape* shape, const int32_t* kept_idx, const int32_t* n_kept,
                   const uint16_t* src, uint16_t* dst, int64_t dst_rows, sp_stream_t stream);

/* Kept token ids for the target's batch (same section): out[i] =
 * token_ids[kept_idx[i]] for i < *n_kept (n_kept read on the device and
 * clamped to [0, n_tokens_total]); an index outside [0, n_tokens_total)
 * gives -1. token_ids holds the packed prompts' ids, n_tokens_total of them;
 * out must hold n_tokens_total entries. All pointers are device pointers.
 * Returns SP_ERR_INVALID_ARG for a null pointer or a bad size. */
int sp_gather_tokens(const int32_t* token_ids, int64_t n_tokens_total, const int32_t* kept_idx,
                     const int32_t* n_kept, int32_t* out, sp_stream_t stream);

/* Keys read in place from a draft engine's cache (in-situ scoring): one
 * key pool per layer, as draft engines allocate them, instead of one
 * [Ly][Ntot][Hk][d] tensor.
 * - layer_k: host array of n_layers (<= 64) device pointers, 16-byte
 *   aligned; pool row r, KV head g, element j of layer l at
 *   layer_k[l][r*k_stride_token + g*k_stride_head + j] (the shape's
 *   k_stride_token and k_stride_head; k_stride_layer is not used).
 * - block_table NULL: pool row = packed token index (seq_off[b] + t);
 *   pool_tokens >= n_tokens_total.
 * - block_table non-NULL (device, [n_seqs][table_stride] int32): a
 *   block-paged cache; token t of prompt b is pool row
 *   block_table[b*table_stride + t/block_size]*block_size + t%block_size.
 *   block_size is 8, 16, 32 or 64, or a multiple of 128; every prompt's
 *   blocks must fit in its table row (else the call's device status is
 *   SP_ERR_DEVICE and nothing is scored); a block id whose rows fall outside
 *   [0, pool_tokens) sets SP_ERR_DEVICE and reads pool row 0 instead.
 * - pool_tokens: rows of each layer's pool (num_blocks * block_size), at
 *   most 2^31 - 1. */
typedef struct sp_kv_source {
    const uint16_t* const* layer_k;
    const int32_t* block_table;
    int32_t block_size;
    int32_t table_stride;
    int64_t pool_tokens;
} sp_kv_source;

/* sp_attn_importance and sp_specprefill_score with the keys from `kv`
 * (the tensor-core path; same outputs, same workspace size for the same
 * shape). */
int sp_attn_importance_kv(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                          const uint16_t* q, const sp_kv_source* kv, float* imp, void* ws,
                          size_t ws_bytes, sp_stream_t stream);
int sp_specprefill_score_kv(const sp_shape* shape, const sp_params* params,
                            const int32_t* seq_off, const uint16_t* q, const sp_kv_source* kv,
                            float* imp, float* tok_score, float* chunk_score, int32_t* chunk_off,
                            uint8_t* chunk_keep, int32_t* kept_idx, int32_t* kept_pos,
                            int32_t* kept_off, int32_t* n_kept, void* ws, size_t ws_bytes,
                            sp_stream_t stream);

/* Sliding-window scoring of the pages' tool ("SpecPrefill — Implementation
 * Guide", v3.1 §Sliding Window Loop and §Bug Fixes in v3.1): a prompt longer
 * than the draft's context is scored in windows of `window` tokens starting
 * every `stride` tokens, each window on its own (its own keys and lookahead
 * queries); window w contributes the scores of its first `stride` tokens,
 * the last window (the first one that reaches the end of the prompt) all of
 * its own, so every token is scored by exactly one window.
 *
 * sp_auto_window (host only): the guide's sizing for a draft context of
 * spec_ctx tokens (v2 listing `main`): a requested window <= 0 becomes
 * min(spec_ctx - 512, 500 MiB / (spec_ctx * 32)), the result is raised to
 * at least 512 and then lowered to at most spec_ctx - 128, and the stride is
 * half of it. SP_ERR_INVALID_ARG when spec_ctx < 130 (the window would be
 * below 2) or an output pointer is null.
 *
 * sp_window_plan (host only): the windows of a prompt of n tokens, in scoring
 * order: window w covers tokens [start[w], end[w]) and contributes its first
 * kept[w] scores. Writes *n_windows; the arrays (host, `capacity` entries
 * each, nullable when capacity is 0) receive min(capacity, *n_windows)
 * windows. SP_ERR_INVALID_ARG unless 1 <= stride <= window and n >= 0.
 *
 * sp_merge_windows (device): out[t] for t < n (device, n floats) from the
 * per-window importance vectors packed back to back in window order
 * (imp_windows, device, sum of the window lengths: every window but the
 * last has `window` tokens), i.e. out[t] = imp_windows[w * window + t -
 * w * stride] with w = min(t / stride, last window). Feed the window batch
 * to sp_attn_importance as a batch of prompts (one per window), merge, then
 * select with sp_select_from_importance. */
int sp_auto_window(int32_t spec_ctx, int32_t window_request, int32_t* window, int32_t* stride);
int sp_window_plan(int64_t n, int32_t window, int32_t stride, int32_t* start, int32_t* end,
                   int32_t* kept, int32_t capacity, int32_t* n_windows);
int sp_merge_windows(int64_t n, int32_t window, int32_t stride, const float* imp_windows,
                     float* out, sp_stream_t stream);

/* Pooling, normalisation, boost, chunk scores, selection and the kept
 * lists from a given per-token importance imp (device, Ntot floats): the
 * part of sp_specprefill_score after the importance, for importance that
 * comes from elsewhere (merged windows, another scorer). `shape` needs only
 * n_seqs and n_tokens_total to be meaningful (the attention dimensions must
 * still pass the checks; sp_workspace_size with the same shape gives the
 * workspace). Outputs as for sp_specprefill_score. */
int sp_select_from_importance(const sp_shape* shape, const sp_params* params,
                              const int32_t* seq_off, const float* imp, float* tok_score,
                              float* chunk_score, int32_t* chunk_off, uint8_t* chunk_keep,
                              int32_t* kept_idx, int32_t* kept_pos, int32_t* kept_off,
                              int32_t* n_kept, void* ws, size_t ws_bytes, sp_stream_t stream);

/* The whole path in one call: sp_attn_importance, sp_pool_chunk, sp_select
 * and sp_gather_kept in sequence, defined by the passages cited at each of
 * them ("SpecPrefill — Implementation Guide", §How It Works / Attention
 * Capture, Token Importance, Sparse Prefill, §Chunk Selection, v3 §v3
 * Improvements items 1-2, v3.1 §v3.1 Optimizations item 5; llama.cpp PR
 * "Speculative prefill", §Approach items 1-4). imp, tok_score, chunk_score, chunk_off and
 * chunk_keep are optional outputs (nullable; kept in the workspace when
 * null); kept_idx, kept_pos, kept_off and n_kept are required. `prof` is
 * optional (nullable). */
int sp_specprefill_score(const sp_shape* shape, const sp_params* params,
                         const int32_t* seq_off, const uint16_t* q, const uint16_t* k,
                         float* imp, float* tok_score, float* chunk_score, int32_t* chunk_off,
                         uint8_t* chunk_keep, int32_t* kept_idx, int32_t* kept_pos,
                         int32_t* kept_off, int32_t* n_kept, void* ws, size_t ws_bytes,
                         sp_stream_t stream, const sp_profile* prof);

/* Synchronise `stream`, then read (and, when `clear` is non-zero, reset)
 * the workspace's sticky device status word into *status_host. */
int sp_get_device_status(void* ws, size_t ws_bytes, sp_stream_t stream, int clear,
                         int32_t* status_host);

/* Static description of a status code. */
const char* sp_status_string(int status);

/* Library build identification (architecture and kernel variant). */
const char* sp_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECPREFILL_H */

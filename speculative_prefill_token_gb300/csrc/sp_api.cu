// C ABI of the SpecPrefill scoring library: argument validation, the
// per-shape launch plan and workspace layout, and the launch sequences of
// the entry points declared in specprefill.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "sp_internal.h"
#include "specprefill.h"

namespace sp {
namespace {

// Default scratch budget of one wave of slabs (quantised logits), unless
// sp_params.wave_mib sets one. Every wave adds a logits-kernel tail and an
// importance kernel between the key streams; measured on GB300, one wave
// whose scratch spills from L2 to HBM (written once, read once) beats two
// L2-sized waves: 258 instead of 295 us per call on the 131K-token d = 128
// workload, 252 instead of 270 on the 16-prompt serving batch; 25 MB for
// the 32K-token 2B workload stays in L2.
constexpr int64_t kWaveScratchBytes = int64_t(2048) << 20;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite_pos(float x) { return std::isfinite(x) && x > 0.0f; }

int check_shape(const sp_shape* s) {
    if (!s) return SP_ERR_INVALID_ARG;
    if (s->n_seqs < 1 || s->n_layers < 1 || s->n_q_heads < 1 || s->n_kv_heads < 1 ||
        s->head_dim < 1 || s->n_lookahead < 1 || s->n_tokens_total < 1 || s->max_seq_len < 0)
        return SP_ERR_INVALID_ARG;
    if (s->n_q_heads % s->n_kv_heads != 0) return SP_ERR_INVALID_ARG;
    if (s->n_seqs > kMaxSeqs) return SP_ERR_UNSUPPORTED;
    if (s->head_dim != 64 && s->head_dim != 128 && s->head_dim != 256) return SP_ERR_UNSUPPORTED;
    const int G = s->n_q_heads / s->n_kv_heads;
    if (static_cast<int64_t>(s->n_lookahead) * G > kMaxRows) return SP_ERR_UNSUPPORTED;
    // strides: positive where the axis has more than one entry, 16-byte multiples
    const int64_t st[7] = {s->k_stride_layer, s->k_stride_token, s->k_stride_head, s->q_stride_seq,
                           s->q_stride_layer, s->q_stride_step, s->q_stride_head};
    const int64_t ext[7] = {s->n_layers, s->n_tokens_total, s->n_kv_heads, s->n_seqs,
                            s->n_layers, s->n_lookahead, s->n_q_heads};
    for (int i = 0; i < 7; ++i) {
        if (ext[i] <= 1) continue;
        if (st[i] < s->head_dim) return SP_ERR_INVALID_ARG;
        if ((st[i] * 2) % 16 != 0) return SP_ERR_UNSUPPORTED;
    }
    if (s->n_tokens_total > (int64_t(1) << 30)) return SP_ERR_UNSUPPORTED;
    return SP_OK;
}

int check_params(const sp_params* p) {
    if (!p) return SP_ERR_INVALID_ARG;
    if (p->pool_w < 1 || p->pool_w % 2 == 0 || p->pool_w > kMaxPool) return SP_ERR_INVALID_ARG;
    if (p->chunk < 1 || p->chunk > kMaxChunk) return SP_ERR_INVALID_ARG;
    if (p->mode != SP_MODE_FIXED && p->mode != SP_MODE_MASS) return SP_ERR_INVALID_ARG;
    if (p->mode == SP_MODE_FIXED && !(finite_pos(p->keep_p) && p->keep_p <= 1.0f)) return SP_ERR_INVALID_ARG;
    if (p->mode == SP_MODE_MASS && !(finite_pos(p->mass) && p->mass <= 1.0f)) return SP_ERR_INVALID_ARG;
    if (!finite_pos(p->boost_first_mult) || !finite_pos(p->boost_last_mult)) return SP_ERR_INVALID_ARG;
    if (p->boost_first_n < 0 || p->boost_last_n < 0) return SP_ERR_INVALID_ARG;
    if (!(std::isfinite(p->scale) && p->scale >= 0.0f)) return SP_ERR_INVALID_ARG;
    if ((p->normalize != 0 && p->normalize != 1) || (p->force_bos != 0 && p->force_bos != 1) ||
        (p->force_last_chunk != 0 && p->force_last_chunk != 1))
        return SP_ERR_INVALID_ARG;
    if ((p->rule != SP_RULE_EXACT && p->rule != SP_RULE_LISTING) || p->min_tok < 0 || p->max_keep < 0)
        return SP_ERR_INVALID_ARG;
    if (p->pool_at != SP_POOL_TOKEN && p->pool_at != SP_POOL_HEAD) return SP_ERR_INVALID_ARG;
    if (p->pool_at == SP_POOL_HEAD && p->pool_w / 2 > 64) return SP_ERR_UNSUPPORTED;
    if (p->wave_mib < 0) return SP_ERR_INVALID_ARG;
    return SP_OK;
}

// The fused post path is available for the parameters the steps after the
// importance see.
bool post_fused(const sp_params* p) {
    const sp_params q = post_params(p);
    return fused_post_ok(&q);
}

int check_ws(const Plan& pl, void* ws, size_t ws_bytes) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < pl.total)
        return SP_ERR_WORKSPACE;
    return SP_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? SP_OK : SP_ERR_CUDA; }

}  // namespace

int make_plan(const sp_shape* s, const sp_params* p, Plan* pl) {
    int rc = check_shape(s);
    if (rc != SP_OK) return rc;
    rc = check_params(p);
    if (rc != SP_OK) return rc;
    Plan& P = *pl;
    std::memset(&P, 0, sizeof(P));
    P.B = s->n_seqs;
    P.Ly = s->n_layers;
    P.Hq = s->n_q_heads;
    P.Hk = s->n_kv_heads;
    P.G = P.Hq / P.Hk;
    P.d = s->head_dim;
    P.L = s->n_lookahead;
    P.R = P.L * P.G;
    P.Rs = P.R <= 32 ? 32 : 64;
    P.Nmma = P.R <= 16 ? 16 : ((P.R + 15) & ~15);
    P.Nacc = P.Nmma <= 32 ? 32 : 64;
    P.Ntot = s->n_tokens_total;
    P.max_len = s->max_seq_len;
    P.slabs = P.Ly * P.Hk;
    P.C = p->chunk;
    P.W = p->pool_w;
    P.tiles_max = P.Ntot / kTileTokens + P.B;
    P.chunks_max = P.Ntot / P.C + P.B;
    P.Tb = P.C <= kPostBlockTarget ? static_cast<int64_t>(P.C) * (kPostBlockTarget / P.C) : P.C;
    P.pblk_max = P.Ntot / P.Tb + P.B;
    P.slices_max = P.chunks_max / kSliceChunks + P.B;
    int64_t maxnc = (P.Ntot + P.C - 1) / P.C;
    if (maxnc > kMaxPromptChunks) maxnc = kMaxPromptChunks;
    P.sort_cap = 1;
    while (P.sort_cap < maxnc) P.sort_cap <<= 1;
    // quantised logits (2 bytes) plus one fp32 maximum per warp quarter and row
    const int64_t per_slab = (P.tiles_max * kTileTokens) * P.Rs * 2 + P.tiles_max * 4 * P.Rs * 4;
    const int64_t budget = p->wave_mib > 0 ? static_cast<int64_t>(p->wave_mib) << 20 : kWaveScratchBytes;
    int64_t spw = budget / per_slab;
    if (spw < 1) spw = 1;
    if (spw > P.slabs) spw = P.slabs;
    {   // the fewest waves the budget allows, of equal size
        const int64_t nw = (P.slabs + spw - 1) / spw;
        spw = (P.slabs + nw - 1) / nw;
    }
    if (spw > 64) spw = 64;
    P.slabs_per_wave = static_cast<int>(spw);
    P.waves = (P.slabs + P.slabs_per_wave - 1) / P.slabs_per_wave;
    // the CUDA-core cross-check runs one item per CTA: up to tiles_max * slabs CTAs
    P.rec_slots = (P.tiles_max * P.slabs_per_wave + static_cast<int64_t>(P.slabs_per_wave) * P.B) * 2;
    const double scale = p->scale > 0.0f ? static_cast<double>(p->scale)
                                          : static_cast<double>(1.0f / std::sqrt(static_cast<float>(P.d)));
    P.scale2 = static_cast<float>(scale * 1.4426950408889634);
    P.spin = p->spin_limit > 0 ? p->spin_limit : kDefaultSpin;
    P.head_h = (p->pool_at == SP_POOL_HEAD && p->pool_w > 1) ? p->pool_w / 2 : 0;

    size_t off = sizeof(WsHeader);
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align256(off + bytes);
        return o;
    };
    const size_t B1 = static_cast<size_t>(P.B) + 1;
    P.o_tile_base = take(B1 * 4);
    P.o_chunk_off = take(B1 * 4);
    P.o_pblk_base = take(B1 * 4);
    P.o_slice_base = take(B1 * 4);
    P.o_scount = take(static_cast<size_t>(P.slices_max) * kRankSplitMax * 4);
    P.o_ucount = take(static_cast<size_t>(P.slices_max) * kRankSplitMax * 4);
    // per-segment record counters, then the listing rule's per-prompt
    // kept counts: one range, zeroed by the prep kernel on every call
    P.o_segcnt = take((static_cast<size_t>(P.slabs_per_wave) + 1) * P.B * 4);
    P.o_lcount = P.o_segcnt + static_cast<size_t>(P.slabs_per_wave) * P.B * 4;
    P.o_logits = take(static_cast<size_t>(P.slabs_per_wave) * P.tiles_max * kTileTokens * P.Rs * 2);
    P.o_lmax = take(static_cast<size_t>(P.slabs_per_wave) * P.tiles_max * 4 * P.Rs * 4);
    P.o_part = take(static_cast<size_t>(P.rec_slots) * P.Rs * 8);
    P.o_lse = take(static_cast<size_t>(P.slabs_per_wave) * P.B * P.Rs * 4);
    P.o_alog = take(P.waves > 1 ? static_cast<size_t>(P.L) * P.Ntot * 4 : 0);
    P.o_imp = take(static_cast<size_t>(P.Ntot) * 4);
    P.o_tok = take(static_cast<size_t>(P.Ntot) * 4);
    P.o_ppart = take(static_cast<size_t>(P.pblk_max) * 8);
    P.o_rpart = take(static_cast<size_t>(P.tiles_max) * 8);  // per 128-token pool CTA
    P.o_csum = take(static_cast<size_t>(P.chunks_max) * 8);
    P.o_cscore = take(static_cast<size_t>(P.chunks_max) * 4);
    P.o_ckeep = take(static_cast<size_t>(P.chunks_max));
    P.o_ckoff = take(static_cast<size_t>(P.chunks_max) * 4);
    P.o_pcount = take(static_cast<size_t>(P.B) * 4);
    P.o_kept_off = take(B1 * 4);
    P.o_nkept = take(4);
    P.total = off;
    return SP_OK;
}

namespace {

int importance_waves(const Plan& pl, const sp_shape* s, const int32_t* seq_off, const uint16_t* q,
                     const uint16_t* k, float* imp, void* ws, cudaStream_t st, bool simt,
                     const sp_profile* prof, const KvSrc* kv = nullptr) {
    if (prof && prof->logits_start)
        if (cudaEventRecord(reinterpret_cast<cudaEvent_t>(prof->logits_start), st) != cudaSuccess)
            return SP_ERR_CUDA;
    for (int w = 0; w < pl.waves; ++w) {
        const int slab0 = w * pl.slabs_per_wave;
        const int ns = pl.slabs - slab0 < pl.slabs_per_wave ? pl.slabs - slab0 : pl.slabs_per_wave;
        int grid = 0;
        cudaError_t e;
        if (simt) {
            e = launch_logits_simt(pl, s, seq_off, q, k, ws, slab0, ns, &grid, st);
        } else {
            grid = logits_tc_grid(pl, ns);
            e = launch_logits_tc(pl, s, seq_off, q, k, ws, slab0, ns, grid, st, kv);
        }
        if (e != cudaSuccess) return SP_ERR_CUDA;
        if (w == pl.waves - 1 && prof && prof->logits_stop)
            if (cudaEventRecord(reinterpret_cast<cudaEvent_t>(prof->logits_stop), st) != cudaSuccess)
                return SP_ERR_CUDA;
        if ((e = launch_reduce(pl, seq_off, ws, ns, w, imp, st)) != cudaSuccess)
            return SP_ERR_CUDA;
    }
    return SP_OK;
}

int attn_importance(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                    const uint16_t* q, const uint16_t* k, float* imp, void* ws, size_t ws_bytes,
                    sp_stream_t stream, bool simt) {
    Plan pl;
    int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !q || !k || !imp || !aligned16(q) || !aligned16(k)) return SP_ERR_INVALID_ARG;
    if ((rc = check_ws(pl, ws, ws_bytes)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (launch_prep(pl, seq_off, ws, nullptr, st) != cudaSuccess) return SP_ERR_CUDA;
    return importance_waves(pl, shape, seq_off, q, k, imp, ws, st, simt, nullptr);
}

// Checks a draft-cache key source, builds the plan (the shape's unused
// layer stride is replaced) and the device-side descriptor.
int kv_plan(const sp_shape* shape, const sp_params* params, const sp_kv_source* kv, sp_shape* s2,
            KvSrc* src, Plan* pl) {
    if (!shape || !kv || !kv->layer_k) return SP_ERR_INVALID_ARG;
    *s2 = *shape;
    s2->k_stride_layer = shape->k_stride_token;  // not used: one pool per layer
    int rc = make_plan(s2, params, pl);
    if (rc != SP_OK) return rc;
    if (pl->Ly > kMaxKvLayers) return SP_ERR_UNSUPPORTED;
    if (kv->pool_tokens < 1 || kv->pool_tokens > INT32_MAX) return SP_ERR_INVALID_ARG;
    std::memset(src, 0, sizeof(*src));
    for (int l = 0; l < pl->Ly; ++l) {
        if (!kv->layer_k[l] || !aligned16(kv->layer_k[l])) return SP_ERR_INVALID_ARG;
        src->layer_k[l] = kv->layer_k[l];
    }
    src->pool_tokens = kv->pool_tokens;
    if (kv->block_table) {
        const int bs = kv->block_size;
        const bool ok_bs = bs == 8 || bs == 16 || bs == 32 || bs == 64 || (bs >= 128 && bs % 128 == 0);
        if (!ok_bs || kv->table_stride < 1) return SP_ERR_INVALID_ARG;
        src->block_table = kv->block_table;
        src->block_size = bs;
        src->table_stride = kv->table_stride;
        pl->kv_block_size = bs;
        pl->kv_table_stride = kv->table_stride;
    } else if (kv->pool_tokens < pl->Ntot) {
        return SP_ERR_INVALID_ARG;
    }
    return SP_OK;
}

// Steps after the importance: pool (+ normalise, boost, chunk sums), chunk
// scores and selection, kept lists. The fused post path when the pool halo
// and chunk size allow it (required by the listing rule), else the staged
// kernels.
int select_tail(const Plan& pl, const sp_params* params, const int32_t* seq_off, const float* imp,
                float* tok_score, float* chunk_score, uint8_t* chunk_keep, int32_t* kept_idx,
                int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept, void* ws, cudaStream_t st) {
    const sp_params pp = post_params(params);
    params = &pp;
    float* tok_p = tok_score ? tok_score : ws_ptr<float>(ws, pl.o_tok);
    float* cs_p = chunk_score ? chunk_score : ws_ptr<float>(ws, pl.o_cscore);
    uint8_t* keep_p = chunk_keep ? chunk_keep : ws_ptr<uint8_t>(ws, pl.o_ckeep);
    const int32_t* coff = ws_ptr<int32_t>(ws, pl.o_chunk_off);
    if (fused_post_ok(params)) {
        if (launch_pool_sums(pl, params, seq_off, imp, tok_p, ws, st) != cudaSuccess)
            return SP_ERR_CUDA;
        return to_status(launch_post(pl, params, seq_off, cs_p, keep_p, kept_idx, kept_pos, kept_off,
                                     n_kept, ws, st));
    }
    if (launch_pool(pl, params, seq_off, imp, tok_p, ws, st) != cudaSuccess) return SP_ERR_CUDA;
    if (launch_chunk(pl, params, seq_off, tok_p, cs_p, ws, st) != cudaSuccess) return SP_ERR_CUDA;
    if (launch_select(pl, params, seq_off, coff, cs_p, keep_p, ws, false, nullptr, nullptr, st) !=
        cudaSuccess)
        return SP_ERR_CUDA;
    if (launch_gather_scan(pl, params, seq_off, coff, keep_p, ws, kept_off, n_kept, st) != cudaSuccess)
        return SP_ERR_CUDA;
    return to_status(launch_gather_write(pl, params, seq_off, coff, keep_p, kept_idx, kept_pos,
                                         kept_off, n_kept, ws, st));
}

}  // namespace
}  // namespace sp

using namespace sp;

extern "C" {

int sp_max_chunks(const sp_shape* shape, const sp_params* params, int64_t* n_chunks) {
    Plan pl;
    const int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!n_chunks) return SP_ERR_INVALID_ARG;
    *n_chunks = pl.chunks_max;
    return SP_OK;
}

int sp_kernels_per_call(const sp_shape* shape, const sp_params* params, int32_t* n_kernels) {
    Plan pl;
    const int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!n_kernels) return SP_ERR_INVALID_ARG;
    // prep, (logits, importance) per wave, then pool sums, rank, gather or
    // pool, chunk, select, gather scan, gather write
    *n_kernels = 1 + 2 * pl.waves + (post_fused(params) ? 3 : 5);
    return SP_OK;
}

int sp_workspace_size(const sp_shape* shape, const sp_params* params, size_t* bytes) {
    Plan pl;
    const int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!bytes) return SP_ERR_INVALID_ARG;
    *bytes = pl.total;
    return SP_OK;
}

int sp_workspace_init(void* ws, size_t ws_bytes, sp_stream_t stream) {
    if (!ws || ws_bytes < sizeof(WsHeader) || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return SP_ERR_WORKSPACE;
    return to_status(cudaMemsetAsync(ws, 0, sizeof(WsHeader), reinterpret_cast<cudaStream_t>(stream)));
}

int sp_attn_importance(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                       const uint16_t* q, const uint16_t* k, float* imp, void* ws, size_t ws_bytes,
                       sp_stream_t stream) {
    return attn_importance(shape, params, seq_off, q, k, imp, ws, ws_bytes, stream, false);
}

int sp_attn_importance_simt(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                            const uint16_t* q, const uint16_t* k, float* imp, void* ws,
                            size_t ws_bytes, sp_stream_t stream) {
    return attn_importance(shape, params, seq_off, q, k, imp, ws, ws_bytes, stream, true);
}

int sp_pool_chunk(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                  const float* imp, float* tok_score, float* chunk_score, int32_t* chunk_off,
                  void* ws, size_t ws_bytes, sp_stream_t stream) {
    Plan pl;
    int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !imp || !chunk_score || !chunk_off) return SP_ERR_INVALID_ARG;
    if ((rc = check_ws(pl, ws, ws_bytes)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* tok = tok_score ? tok_score : ws_ptr<float>(ws, pl.o_tok);
    if (launch_prep(pl, seq_off, ws, chunk_off, st) != cudaSuccess) return SP_ERR_CUDA;
    const sp_params pp = post_params(params);
    if (launch_pool(pl, &pp, seq_off, imp, tok, ws, st) != cudaSuccess) return SP_ERR_CUDA;
    return to_status(launch_chunk(pl, &pp, seq_off, tok, chunk_score, ws, st));
}

int sp_select(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
              const int32_t* chunk_off, const float* chunk_score, uint8_t* chunk_keep, void* ws,
              size_t ws_bytes, sp_stream_t stream) {
    Plan pl;
    int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !chunk_off || !chunk_score || !chunk_keep) return SP_ERR_INVALID_ARG;
    if (params->rule != SP_RULE_EXACT) return SP_ERR_UNSUPPORTED;
    if ((rc = check_ws(pl, ws, ws_bytes)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (launch_prep_check(pl, seq_off, ws, chunk_off, st) != cudaSuccess) return SP_ERR_CUDA;
    return to_status(launch_select(pl, params, seq_off, ws_ptr<int32_t>(ws, pl.o_chunk_off),
                                   chunk_score, chunk_keep, ws, false, nullptr, nullptr, st));
}

int sp_gather_kept(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                   const int32_t* chunk_off, const uint8_t* chunk_keep, int32_t* kept_idx,
                   int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept, void* ws, size_t ws_bytes,
                   sp_stream_t stream) {
    Plan pl;
    int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !chunk_off || !chunk_keep || !kept_idx || !kept_pos || !kept_off || !n_kept)
        return SP_ERR_INVALID_ARG;
    if (params->rule != SP_RULE_EXACT) return SP_ERR_UNSUPPORTED;
    if ((rc = check_ws(pl, ws, ws_bytes)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int32_t* coff = ws_ptr<int32_t>(ws, pl.o_chunk_off);
    if (launch_prep_check(pl, seq_off, ws, chunk_off, st) != cudaSuccess) return SP_ERR_CUDA;
    if (launch_gather_scan(pl, params, seq_off, coff, chunk_keep, ws, kept_off, n_kept, st) !=
        cudaSuccess)
        return SP_ERR_CUDA;
    return to_status(launch_gather_write(pl, params, seq_off, coff, chunk_keep, kept_idx, kept_pos,
                                         kept_off, n_kept, ws, st));
}

int sp_specprefill_score(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                         const uint16_t* q, const uint16_t* k, float* imp, float* tok_score,
                         float* chunk_score, int32_t* chunk_off, uint8_t* chunk_keep,
                         int32_t* kept_idx, int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept,
                         void* ws, size_t ws_bytes, sp_stream_t stream, const sp_profile* prof) {
    Plan pl;
    int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !q || !k || !kept_idx || !kept_pos || !kept_off || !n_kept || !aligned16(q) ||
        !aligned16(k))
        return SP_ERR_INVALID_ARG;
    if (params->rule != SP_RULE_EXACT && !post_fused(params)) return SP_ERR_UNSUPPORTED;
    if ((rc = check_ws(pl, ws, ws_bytes)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* imp_p = imp ? imp : ws_ptr<float>(ws, pl.o_imp);
    if (launch_prep(pl, seq_off, ws, chunk_off, st) != cudaSuccess) return SP_ERR_CUDA;
    if ((rc = importance_waves(pl, shape, seq_off, q, k, imp_p, ws, st, false, prof)) != SP_OK)
        return rc;
    return select_tail(pl, params, seq_off, imp_p, tok_score, chunk_score, chunk_keep, kept_idx,
                       kept_pos, kept_off, n_kept, ws, st);
}

int sp_select_from_importance(const sp_shape* shape, const sp_params* params,
                              const int32_t* seq_off, const float* imp, float* tok_score,
                              float* chunk_score, int32_t* chunk_off, uint8_t* chunk_keep,
                              int32_t* kept_idx, int32_t* kept_pos, int32_t* kept_off,
                              int32_t* n_kept, void* ws, size_t ws_bytes, sp_stream_t stream) {
    Plan pl;
    int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !imp || !kept_idx || !kept_pos || !kept_off || !n_kept) return SP_ERR_INVALID_ARG;
    if (params->rule != SP_RULE_EXACT && !post_fused(params)) return SP_ERR_UNSUPPORTED;
    if ((rc = check_ws(pl, ws, ws_bytes)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (launch_prep(pl, seq_off, ws, chunk_off, st) != cudaSuccess) return SP_ERR_CUDA;
    return select_tail(pl, params, seq_off, imp, tok_score, chunk_score, chunk_keep, kept_idx,
                       kept_pos, kept_off, n_kept, ws, st);
}

int sp_attn_importance_kv(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                          const uint16_t* q, const sp_kv_source* kv, float* imp, void* ws,
                          size_t ws_bytes, sp_stream_t stream) {
    sp_shape s2;
    KvSrc src;
    Plan pl;
    int rc = kv_plan(shape, params, kv, &s2, &src, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !q || !imp || !aligned16(q)) return SP_ERR_INVALID_ARG;
    if ((rc = check_ws(pl, ws, ws_bytes)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (launch_prep(pl, seq_off, ws, nullptr, st) != cudaSuccess) return SP_ERR_CUDA;
    return importance_waves(pl, &s2, seq_off, q, nullptr, imp, ws, st, false, nullptr, &src);
}

int sp_specprefill_score_kv(const sp_shape* shape, const sp_params* params, const int32_t* seq_off,
                            const uint16_t* q, const sp_kv_source* kv, float* imp, float* tok_score,
                            float* chunk_score, int32_t* chunk_off, uint8_t* chunk_keep,
                            int32_t* kept_idx, int32_t* kept_pos, int32_t* kept_off, int32_t* n_kept,
                            void* ws, size_t ws_bytes, sp_stream_t stream) {
    sp_shape s2;
    KvSrc src;
    Plan pl;
    int rc = kv_plan(shape, params, kv, &s2, &src, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !q || !kept_idx || !kept_pos || !kept_off || !n_kept || !aligned16(q))
        return SP_ERR_INVALID_ARG;
    if (params->rule != SP_RULE_EXACT && !post_fused(params)) return SP_ERR_UNSUPPORTED;
    if ((rc = check_ws(pl, ws, ws_bytes)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* imp_p = imp ? imp : ws_ptr<float>(ws, pl.o_imp);
    if (launch_prep(pl, seq_off, ws, chunk_off, st) != cudaSuccess) return SP_ERR_CUDA;
    if ((rc = importance_waves(pl, &s2, seq_off, q, nullptr, imp_p, ws, st, false, nullptr, &src)) != SP_OK)
        return rc;
    return select_tail(pl, params, seq_off, imp_p, tok_score, chunk_score, chunk_keep, kept_idx,
                       kept_pos, kept_off, n_kept, ws, st);
}

int sp_auto_window(int32_t spec_ctx, int32_t window_request, int32_t* window, int32_t* stride) {
    if (!window || !stride || spec_ctx < 130) return SP_ERR_INVALID_ARG;
    const int64_t max_safe = (int64_t(500) * 1024 * 1024) / (static_cast<int64_t>(spec_ctx) * 32);
    int64_t w = window_request;
    if (w <= 0) w = std::min<int64_t>(spec_ctx - 512, max_safe);
    w = std::max<int64_t>(w, 512);
    w = std::min<int64_t>(w, spec_ctx - 128);
    *window = static_cast<int32_t>(w);
    *stride = static_cast<int32_t>(w / 2);
    return SP_OK;
}

int sp_window_plan(int64_t n, int32_t window, int32_t stride, int32_t* start, int32_t* end,
                   int32_t* kept, int32_t capacity, int32_t* n_windows) {
    if (!n_windows || n < 0 || n > (int64_t(1) << 30) || stride < 1 || window < stride ||
        capacity < 0 || (capacity > 0 && (!start || !end || !kept)))
        return SP_ERR_INVALID_ARG;
    int32_t w = 0;
    for (int64_t pos = 0; pos < n; pos += stride) {
        const int64_t e = std::min<int64_t>(pos + window, n);
        const bool last = e >= n || pos + stride >= n;
        if (w < capacity) {
            start[w] = static_cast<int32_t>(pos);
            end[w] = static_cast<int32_t>(e);
            kept[w] = static_cast<int32_t>(last ? e - pos : stride);
        }
        ++w;
        if (last) break;
    }
    *n_windows = w;
    return SP_OK;
}

int sp_merge_windows(int64_t n, int32_t window, int32_t stride, const float* imp_windows,
                     float* out, sp_stream_t stream) {
    if (!imp_windows || !out || n < 0 || n > (int64_t(1) << 30) || stride < 1 || window < stride)
        return SP_ERR_INVALID_ARG;
    if (n == 0) return SP_OK;
    return to_status(launch_merge_windows(n, window, stride, imp_windows, out,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int sp_gather_rows(const sp_shape* shape, const int32_t* kept_idx, const int32_t* n_kept,
                   const uint16_t* src, uint16_t* dst, int64_t dst_rows, sp_stream_t stream) {
    if (!shape || !kept_idx || !n_kept || !src || !dst) return SP_ERR_INVALID_ARG;
    const sp_shape* s = shape;
    if (s->n_layers < 1 || s->n_kv_heads < 1 || s->head_dim < 8 || s->head_dim % 8 != 0 ||
        s->n_tokens_total < 1 || s->n_tokens_total > (int64_t(1) << 30) ||
        dst_rows < s->n_tokens_total)
        return SP_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return SP_ERR_INVALID_ARG;
    const int64_t st[3] = {s->k_stride_layer, s->k_stride_token, s->k_stride_head};
    const int64_t ext[3] = {s->n_layers, s->n_tokens_total, s->n_kv_heads};
    for (int i = 0; i < 3; ++i) {
        if (ext[i] <= 1) continue;
        if (st[i] < s->head_dim || st[i] % 8 != 0) return SP_ERR_INVALID_ARG;
    }
    return to_status(launch_gather_rows(s, kept_idx, n_kept, src, dst, dst_rows,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int sp_gather_tokens(const int32_t* token_ids, int64_t n_tokens_total, const int32_t* kept_idx,
                     const int32_t* n_kept, int32_t* out, sp_stream_t stream) {
    if (!token_ids || !kept_idx || !n_kept || !out || n_tokens_total < 1 ||
        n_tokens_total > (int64_t(1) << 30))
        return SP_ERR_INVALID_ARG;
    return to_status(launch_gather_tokens(token_ids, kept_idx, n_kept, out, n_tokens_total,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int sp_get_device_status(void* ws, size_t ws_bytes, sp_stream_t stream, int clear,
                         int32_t* status_host) {
    if (!ws || ws_bytes < sizeof(WsHeader) || !status_host) return SP_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SP_ERR_CUDA;
    if (cudaMemcpy(status_host, ws, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SP_ERR_CUDA;
    if (clear && cudaMemset(ws, 0, sizeof(int32_t)) != cudaSuccess) return SP_ERR_CUDA;
    return SP_OK;
}

const char* sp_status_string(int status) {
    switch (status) {
        case SP_OK: return "ok";
        case SP_ERR_INVALID_ARG: return "invalid argument";
        case SP_ERR_UNSUPPORTED: return "unsupported shape or layout";
        case SP_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case SP_ERR_CUDA: return "CUDA runtime or launch error";
        case SP_ERR_TIMEOUT: return "a bounded device wait gave up";
        case SP_ERR_DEVICE: return "device-side input check failed";
        default: return "unknown status";
    }
}

const char* sp_build_info(void) {
    return "specprefill sm_103a: tcgen05/TMA logits kernel, 16-bit fixed-point logits scratch, "
           "slice-parallel chunk ranking, kept-row gathers";
}

}  // extern "C"

// Token importance with per-head pooling: the variant of the SpecPrefill
// scoring path where the W-wide average pool smooths every attention row
// before the max over heads and layers (llama.cpp PR "Speculative prefill"
// §Approach item 3 lists the smoothing with the max-reduction across
// heads/layers; this is the reading that pools first).
//
// Same inputs as the importance kernel: the quantised logits scratch of a
// wave of slabs (16-bit steps of 2^-11 below the warp-quarter row maximum),
// the per-quarter row maxima and the per-(slab, prompt) log2 normalisers.
// One CTA scores TOK consecutive tokens of one prompt (TOK = 64 for 32 rows
// per slab, 32 for 64). For every slab of the wave it
//   1. converts the quantised values of its tokens plus a halo of W/2 on
//      each side (clipped to the prompt) into probabilities in shared
//      memory, p = exp2(M - q 2^-11 - lse2), zero outside the prompt;
//   2. pools each row: the sum over the window divided by the number of
//      window positions inside the prompt. The tile is stored row-major
//      ([row][token], stride = 4 mod 8 floats), so each thread reads its
//      row's first window with 16-byte loads and slides it over a run of 8
//      outputs (one load in, one value out per step);
//   3. keeps the running maximum per (token, row).
// The next slab's values and maxima are loaded while the current one is
// pooled. After the wave, the maximum over the query heads of each
// lookahead step is combined with the earlier waves' (linear values here)
// and the last wave writes imp = the mean over the steps.
#include <cuda_runtime.h>

#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_phases.cuh"

namespace sp {
namespace {

constexpr int kHpThreads = 256;
constexpr int kHpMaxTab = 2;     // per-quarter offsets per thread and slab (quarters * Rs / 256)
constexpr int kHpRun = 8;        // consecutive outputs of one row per thread

struct HeadPoolArgs {
    const uint16_t* logits;
    const float* lmax;
    const float* lse2;
    const int32_t* seq_off;
    const int32_t* tile_base;
    float* alog;
    float* imp;
    const int32_t* bad;
    int64_t Ntot, rows_per_slab, tiles_max;
    int B, G, L, Rs, nslab, H, first_wave, last_wave;
};

// Tokens per CTA, the probability tile's row stride (>= the halo-extended
// token count E, = 4 mod 8 floats, so that 32 rows read with 16-byte loads
// hit distinct banks) and the CTA's shared-memory floats: the per-quarter
// offset table, then the tile [Rs][stride] (reused for the per-token maxima
// [TOK][Rs + 1] at the end).
__host__ __device__ inline int hp_tok(int Rs) { return kHpThreads / (Rs / 8); }
__host__ __device__ inline int hp_quarters(int Rs, int H) { return (hp_tok(Rs) + 2 * H + 31) / 32 + 1; }
__host__ __device__ inline int hp_stride(int Rs, int H) {
    const int E = hp_tok(Rs) + 2 * H;
    return E + ((12 - E % 8) % 8);
}
__host__ __device__ inline int hp_smem_floats(int Rs, int H) {
    const int tile = Rs * hp_stride(Rs, H), ms = hp_tok(Rs) * (Rs + 1);
    return hp_quarters(Rs, H) * Rs + (tile > ms ? tile : ms);
}

template <int RS>
__global__ void __launch_bounds__(kHpThreads, 4) reduce_head_pool_kernel(const HeadPoolArgs a) {
    constexpr int Q8 = RS / 8, TOK = kHpThreads / Q8, RS1 = RS + 1;
    // 16-byte scratch loads per thread and slab: ceil(E / 32) * 32 tokens x Q8 (W / 2 <= 64)
    constexpr int kItems = ((TOK + 128 + 31) / 32 * 32 * Q8 + kHpThreads - 1) / kHpThreads;
    grid_dep_wait();
    grid_dep_launch();
    const int subs = kTileTokens / TOK;
    const int64_t tile = blockIdx.x / subs;
    const int sub = static_cast<int>(blockIdx.x - tile * subs);
    // the tile's prompt: from Ntot for a single prompt (the prep kernel
    // rejects offsets other than {0, Ntot}), else one round of loads
    Located<1> loc;
    if (a.B == 1) {
        const int64_t hi[1] = {a.Ntot};
        loc = one_prompt<1>(static_cast<int32_t>((a.Ntot + kTileTokens - 1) / kTileTokens), hi);
    } else {
        const int32_t* const aux[1] = {a.seq_off};
        loc = locate<1>(a.tile_base, aux, a.B, tile);
    }
    if (*a.bad) return;
    if (tile >= loc.total) return;
    const int b = loc.b;
    const int64_t base_b = loc.base_b;
    const int64_t start = loc.lo[0];
    const int64_t n = static_cast<int64_t>(loc.hi[0]) - start;
    const int64_t first = (tile - base_b) * kTileTokens + static_cast<int64_t>(sub) * TOK;
    const int nvalid = static_cast<int>(min64(TOK, n - first));
    if (nvalid <= 0) return;
    const int H = a.H, E = TOK + 2 * H, S = hp_stride(RS, H);
    const int n_items = (E + 31) / 32 * 32 * Q8;
    const int64_t e0 = first - H;                              // prompt index of halo token 0
    const int64_t e_lo = max64(e0, 0), e_hi = min64(first + TOK + H, n);
    const int64_t pq_lo = e_lo / 32;                           // first prompt quarter covered
    const int nqe = static_cast<int>((e_hi - 1) / 32 - pq_lo + 1);
    extern __shared__ float sm[];
    float* tab = sm;                                           // [nqe][RS]: M - lse2
    float* P = tab + hp_quarters(RS, H) * RS;                  // [RS][S]: p of row r, halo token e
    const int64_t row0 = base_b * kTileTokens;  // scratch row of token 0
    const int t = threadIdx.x;
    const int n_tab = nqe * RS;

    // item it: 16 bytes (rows 8 cc .. 8 cc + 7) of halo token e; the 32
    // lanes of a warp take 32 consecutive tokens of one row group, so that
    // their shared-memory stores (P[row][e]) hit distinct banks
    uint4 vq[kItems];
    float tl[kHpMaxTab], ts[kHpMaxTab];
    auto load_slab = [&](int s) {
        const uint16_t* base = a.logits + (static_cast<int64_t>(s) * a.rows_per_slab + row0) * RS;
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int it = t + j * kHpThreads, wi = it >> 5;
            const int cc = wi % Q8, e = (wi / Q8) * 32 + (it & 31);
            const int64_t pt = e0 + e;
            vq[j] = make_uint4(0, 0, 0, 0);
            if (it < n_items && e < E && pt >= 0 && pt < n)
                vq[j] = __ldcs(reinterpret_cast<const uint4*>(base + pt * RS + 8 * cc));
        }
#pragma unroll
        for (int j = 0; j < kHpMaxTab; ++j) {
            const int idx = t + j * kHpThreads;
            tl[j] = 0.0f;
            ts[j] = 0.0f;
            if (idx < n_tab) {
                const int qq = idx / RS, r = idx - qq * RS;
                const int64_t pq = pq_lo + qq;
                const int64_t gt = base_b + pq / 4;
                tl[j] = __ldcg(a.lmax + ((static_cast<int64_t>(s) * a.tiles_max + gt) * 4 + pq % 4) * RS + r);
                ts[j] = __ldcg(a.lse2 + (static_cast<int64_t>(s) * a.B + b) * RS + r);
            }
        }
    };

    // pooling role: row pr, outputs tq0 .. tq0 + kHpRun - 1 (their windows
    // are halo tokens tq0 + k .. tq0 + k + 2H)
    const int pr = t % RS, tq0 = (t / RS) * kHpRun;
    const float* prow = P + pr * S + tq0;
    float inv[kHpRun], m[kHpRun];
#pragma unroll
    for (int k = 0; k < kHpRun; ++k) {
        const int64_t pt = first + tq0 + k;
        const int64_t cnt = min64(n, pt + H + 1) - max64(0, pt - H);
        inv[k] = cnt > 0 ? 1.0f / static_cast<float>(cnt) : 0.0f;
        m[k] = 0.0f;
    }

    load_slab(0);
    for (int s = 0; s < a.nslab; ++s) {
#pragma unroll
        for (int j = 0; j < kHpMaxTab; ++j) {
            const int idx = t + j * kHpThreads;
            if (idx < n_tab) tab[idx] = tl[j] - ts[j];
        }
        __syncthreads();  // the table is complete; the previous slab's P is no longer read
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int it = t + j * kHpThreads, wi = it >> 5;
            const int cc = wi % Q8, e = (wi / Q8) * 32 + (it & 31);
            if (it < n_items && e < E) {
                const int64_t pt = e0 + e;
                float* dst = P + (8 * cc) * S + e;
                if (pt >= 0 && pt < n) {
                    const float* off = tab + (pt / 32 - pq_lo) * RS + 8 * cc;
                    const uint32_t w[4] = {vq[j].x, vq[j].y, vq[j].z, vq[j].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        dst[(2 * k) * S] = exp2_ftz(fmaf(-static_cast<float>(w[k] & 0xffffu), kLogitQuantInv, off[2 * k]));
                        dst[(2 * k + 1) * S] = exp2_ftz(fmaf(-static_cast<float>(w[k] >> 16), kLogitQuantInv, off[2 * k + 1]));
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) dst[k * S] = 0.0f;
                }
            }
        }
        if (s + 1 < a.nslab) load_slab(s + 1);
        __syncthreads();  // P complete
        {
            // first window: halo tokens 0 .. 2H of the run, 16-byte loads
            const float4 c0 = *reinterpret_cast<const float4*>(prow);
            const float4 c1 = *reinterpret_cast<const float4*>(prow + 4);
            const float v[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            float sum = 0.0f;
#pragma unroll
            for (int u = 0; u < 8; ++u) sum += u <= 2 * H ? v[u] : 0.0f;
            for (int u = 8; u <= 2 * H; u += 4) {
                const float4 c = *reinterpret_cast<const float4*>(prow + u);
                sum += c.x + (u + 1 <= 2 * H ? c.y : 0.0f) + (u + 2 <= 2 * H ? c.z : 0.0f) +
                       (u + 3 <= 2 * H ? c.w : 0.0f);
            }
            m[0] = fmaxf(m[0], sum * inv[0]);
            // slide: add halo token k + 2H, drop token k - 1
#pragma unroll
            for (int k = 1; k < kHpRun; ++k) {
                sum += prow[k + 2 * H] - v[k - 1];
                m[k] = fmaxf(m[k], sum * inv[k]);
            }
        }
    }
    __syncthreads();  // P is reused for the per-token maxima
    float* ms = P;    // [TOK][RS + 1]
#pragma unroll
    for (int k = 0; k < kHpRun; ++k) ms[(tq0 + k) * RS1 + pr] = m[k];
    __syncthreads();
    if (t < nvalid) {
        const int64_t tok = start + first + t;
        const float* mrow = ms + t * RS1;
        float total = 0.0f;
        for (int l = 0; l < a.L; ++l) {
            float v = 0.0f;
            for (int j = 0; j < a.G; ++j) v = fmaxf(v, mrow[l * a.G + j]);
            if (!a.first_wave) v = fmaxf(v, a.alog[l * a.Ntot + tok]);
            if (a.last_wave) total += v;
            else a.alog[l * a.Ntot + tok] = v;
        }
        if (a.last_wave) a.imp[tok] = total / static_cast<float>(a.L);
    }
}

}  // namespace

size_t head_pool_smem(int Rs, int H) { return sizeof(float) * static_cast<size_t>(hp_smem_floats(Rs, H)); }

cudaError_t launch_reduce_head_pool(const Plan& pl, const int32_t* seq_off, void* ws, int nslab,
                                    int wave, float* imp, cudaStream_t st) {
    HeadPoolArgs a;
    a.logits = ws_ptr<uint16_t>(ws, pl.o_logits);
    a.lmax = ws_ptr<float>(ws, pl.o_lmax);
    a.lse2 = ws_ptr<float>(ws, pl.o_lse);
    a.seq_off = seq_off;
    a.tile_base = ws_ptr<int32_t>(ws, pl.o_tile_base);
    a.alog = ws_ptr<float>(ws, pl.o_alog);
    a.imp = imp;
    a.bad = &ws_ptr<WsHeader>(ws, 0)->bad_input;
    a.Ntot = pl.Ntot;
    a.rows_per_slab = pl.tiles_max * kTileTokens;
    a.tiles_max = pl.tiles_max;
    a.B = pl.B;
    a.G = pl.G;
    a.L = pl.L;
    a.Rs = pl.Rs;
    a.nslab = nslab;
    a.H = pl.head_h;
    a.first_wave = wave == 0 ? 1 : 0;
    a.last_wave = wave == pl.waves - 1 ? 1 : 0;
    const size_t smem = head_pool_smem(pl.Rs, pl.head_h);
    auto kern = pl.Rs == 32 ? reduce_head_pool_kernel<32> : reduce_head_pool_kernel<64>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const unsigned grid = static_cast<unsigned>(pl.tiles_max * (kTileTokens / hp_tok(pl.Rs)));
    return launch_k(kern, grid, kHpThreads, smem, st, a);
}

}  // namespace sp

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
//      window positions inside the prompt;
//   3. keeps the running maximum per (token, row).
// The next slab's values and maxima are loaded while the current one is
// pooled. After the wave, the maximum over the query heads of each
// lookahead step is combined with the earlier waves' (linear values here)
// and the last wave writes imp = the mean over the steps.
#include <cuda_runtime.h>

#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {
namespace {

constexpr int kHpThreads = 256;
constexpr int kHpMaxItems = 6;   // 16-byte scratch loads per thread and slab (E * Rs / 8 / 256)
constexpr int kHpMaxTab = 2;     // per-quarter offsets per thread and slab (quarters * Rs / 256)

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

// Shared-memory floats of one CTA: the per-quarter offset table and the
// probability tile (also reused for the per-token maxima at the end).
__host__ __device__ inline int hp_tok(int Rs) { return kHpThreads / (Rs / 8); }
__host__ __device__ inline int hp_quarters(int Rs, int H) { return (hp_tok(Rs) + 2 * H + 31) / 32 + 1; }
__host__ __device__ inline int hp_smem_floats(int Rs, int H) {
    const int E = hp_tok(Rs) + 2 * H;
    return hp_quarters(Rs, H) * Rs + E * (Rs + 1);
}

__global__ void __launch_bounds__(kHpThreads) reduce_head_pool_kernel(const HeadPoolArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    const int Rs = a.Rs, Q8 = Rs / 8, TOK = hp_tok(Rs), RS1 = Rs + 1;
    const int subs = kTileTokens / TOK;
    const int64_t tile = blockIdx.x / subs;
    const int sub = static_cast<int>(blockIdx.x - tile * subs);
    if (*a.bad) return;
    if (tile >= a.tile_base[a.B]) return;
    const int b = search_base(a.tile_base, a.B, tile);
    const int64_t start = a.seq_off[b];
    const int64_t n = static_cast<int64_t>(a.seq_off[b + 1]) - start;
    const int64_t first = (tile - a.tile_base[b]) * kTileTokens + static_cast<int64_t>(sub) * TOK;
    const int nvalid = static_cast<int>(min64(TOK, n - first));
    if (nvalid <= 0) return;
    const int H = a.H, E = TOK + 2 * H;
    const int64_t e0 = first - H;                              // prompt index of halo token 0
    const int64_t e_lo = max64(e0, 0), e_hi = min64(first + TOK + H, n);
    const int64_t pq_lo = e_lo / 32;                           // first prompt quarter covered
    const int nqe = static_cast<int>((e_hi - 1) / 32 - pq_lo + 1);
    extern __shared__ float sm[];
    float* tab = sm;                                           // [nqe][Rs]: M - lse2
    float* P = tab + hp_quarters(Rs, H) * Rs;                  // [E][Rs + 1]
    const int64_t row0 = static_cast<int64_t>(a.tile_base[b]) * kTileTokens;  // scratch row of token 0
    const int t = threadIdx.x;
    const int n_items = E * Q8, n_tab = nqe * Rs;

    uint4 vq[kHpMaxItems];
    float tl[kHpMaxTab], ts[kHpMaxTab];
    auto load_slab = [&](int s) {
        const uint16_t* base = a.logits + (static_cast<int64_t>(s) * a.rows_per_slab + row0) * Rs;
#pragma unroll
        for (int j = 0; j < kHpMaxItems; ++j) {
            const int it = t + j * kHpThreads;
            vq[j] = make_uint4(0, 0, 0, 0);
            if (it < n_items) {
                const int e = it / Q8, cc = it - e * Q8;
                const int64_t pt = e0 + e;
                if (pt >= 0 && pt < n)
                    vq[j] = __ldcs(reinterpret_cast<const uint4*>(base + pt * Rs + 8 * cc));
            }
        }
#pragma unroll
        for (int j = 0; j < kHpMaxTab; ++j) {
            const int idx = t + j * kHpThreads;
            tl[j] = 0.0f;
            ts[j] = 0.0f;
            if (idx < n_tab) {
                const int qq = idx / Rs, r = idx - qq * Rs;
                const int64_t pq = pq_lo + qq;
                const int64_t gt = a.tile_base[b] + pq / 4;
                tl[j] = __ldcg(a.lmax + ((static_cast<int64_t>(s) * a.tiles_max + gt) * 4 + pq % 4) * Rs + r);
                ts[j] = __ldcg(a.lse2 + (static_cast<int64_t>(s) * a.B + b) * Rs + r);
            }
        }
    };

    const int tq = t / Q8, c = t - tq * Q8;
    const bool act = tq < nvalid;
    const int64_t pt_out = first + tq;
    const float inv_cnt = 1.0f / static_cast<float>(min64(n, pt_out + H + 1) - max64(0, pt_out - H));
    float m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = 0.0f;

    load_slab(0);
    for (int s = 0; s < a.nslab; ++s) {
#pragma unroll
        for (int j = 0; j < kHpMaxTab; ++j) {
            const int idx = t + j * kHpThreads;
            if (idx < n_tab) tab[idx] = tl[j] - ts[j];
        }
        __syncthreads();  // the table is complete; the previous slab's P is no longer read
#pragma unroll
        for (int j = 0; j < kHpMaxItems; ++j) {
            const int it = t + j * kHpThreads;
            if (it < n_items) {
                const int e = it / Q8, cc = it - e * Q8;
                const int64_t pt = e0 + e;
                float* dst = P + e * RS1 + 8 * cc;
                if (pt >= 0 && pt < n) {
                    const float* off = tab + (pt / 32 - pq_lo) * Rs + 8 * cc;
                    const uint32_t w[4] = {vq[j].x, vq[j].y, vq[j].z, vq[j].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        dst[2 * k] = exp2f(fmaf(-static_cast<float>(w[k] & 0xffffu), kLogitQuantInv, off[2 * k]));
                        dst[2 * k + 1] = exp2f(fmaf(-static_cast<float>(w[k] >> 16), kLogitQuantInv, off[2 * k + 1]));
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) dst[k] = 0.0f;
                }
            }
        }
        if (s + 1 < a.nslab) load_slab(s + 1);
        __syncthreads();  // P complete
        if (act) {
            float acc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
            const float* col = P + tq * RS1 + 8 * c;
            for (int o = 0; o <= 2 * H; ++o) {
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] += col[o * RS1 + k];
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], acc[k] * inv_cnt);
        }
    }
    __syncthreads();  // P is reused for the per-token maxima
    float* ms = P;    // [TOK][Rs + 1]
    if (act) {
#pragma unroll
        for (int k = 0; k < 8; ++k) ms[tq * RS1 + 8 * c + k] = m[k];
    }
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
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(reduce_head_pool_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const unsigned grid = static_cast<unsigned>(pl.tiles_max * (kTileTokens / hp_tok(pl.Rs)));
    return launch_k(reduce_head_pool_kernel, grid, kHpThreads, smem, st, a);
}

}  // namespace sp

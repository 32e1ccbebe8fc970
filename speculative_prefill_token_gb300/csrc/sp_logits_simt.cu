// CUDA-core (FP32 FMA) variant of the logits kernel. Same contract and
// quantised scratch format as the tensor-core kernel: one CTA per (128-token tile,
// slab), one thread per key, fp32 accumulation of the R dot products
// against queries staged in shared memory. It is the independent
// cross-check of the tensor-core kernel in the GPU tests; the library's
// entry points always run the tensor-core kernel.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {
namespace {

struct SimtArgs {
    const int32_t* seq_off;
    const int32_t* tile_base;
    const uint16_t* q;
    const uint16_t* k;
    uint16_t* logits;  // [nslab][tiles_max * 128][Rs], quantised scaled logits
    float* lmax;       // [nslab][tiles_max][4][Rs] warp-quarter row maxima
    float2* rec;     // softmax records [(cta + segment) * 2 + warpgroup][Rs]
    unsigned* seg_cnt;
    float* lse2;
    const int32_t* bad;
    int B, Hk, G, L, R, Rs, d, slab0, nslab;
    int64_t rows_per_slab, tiles_max;
    int64_t ks_layer, ks_token, ks_head, qs_seq, qs_layer, qs_step, qs_head;
    float scale2;
};

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// One work item (tile of one slab) per CTA; CTAs past the last item exit.
template <int NH>
__global__ void __launch_bounds__(128) logits_simt_kernel(const SimtArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    if (*a.bad) return;
    constexpr int RMAX = 32 * NH;
    const int64_t T = a.tile_base[a.B];
    const int64_t W = T * a.nslab;
    const int64_t w0 = split_start(W, gridDim.x, blockIdx.x);
    const int64_t w1 = split_start(W, gridDim.x, blockIdx.x + 1);
    if (w0 >= w1) return;
    extern __shared__ float qs[];  // [RMAX][d]
    __shared__ float2 stats[4 * 64];
    __shared__ int seg_flag;
    const int slab_local = static_cast<int>(w0 / T);
    const int64_t tile = w0 - static_cast<int64_t>(slab_local) * T;
    const int b = search_base(a.tile_base, a.B, tile);
    const int64_t i = tile - a.tile_base[b];
    const int64_t start = a.seq_off[b];
    const int64_t n = static_cast<int64_t>(a.seq_off[b + 1]) - start;
    const int64_t tok0 = start + i * kTileTokens;
    const int nvalid = static_cast<int>(min64(kTileTokens, n - i * kTileTokens));
    const int slab = a.slab0 + slab_local;
    const int layer = slab / a.Hk, g = slab - layer * a.Hk;

    for (int idx = threadIdx.x; idx < RMAX * a.d; idx += blockDim.x) {
        const int r = idx / a.d, x = idx - r * a.d;
        float v = 0.0f;
        if (r < a.R) {
            const int s = r / a.G, h = g * a.G + (r - s * a.G);
            v = bf16_to_f32(a.q[b * a.qs_seq + layer * a.qs_layer + s * a.qs_step + h * a.qs_head + x]);
        }
        qs[idx] = v;
    }
    __syncthreads();

    const int t = threadIdx.x;
    const bool valid = t < nvalid;
    float v[NH][32];
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int r = 0; r < 32; ++r) v[h][r] = 0.0f;
    if (valid) {
        const uint16_t* krow = a.k + layer * a.ks_layer + (tok0 + t) * a.ks_token + g * a.ks_head;
        for (int x0 = 0; x0 < a.d; x0 += 8) {
            const uint4 raw = *reinterpret_cast<const uint4*>(krow + x0);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            float kf[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kf[2 * e] = __uint_as_float(w[e] << 16);
                kf[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const float* qr = qs + (h * 32 + r) * a.d + x0;
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[h][r] = fmaf(kf[e], qr[e], v[h][r]);
                }
        }
    }
    RowStats<NH> rs;
    stats_reset(rs);
    if (valid) stats_add<NH>(rs, v, a.scale2);
    // quantised scratch, same format as the tensor-core kernel: row maxima
    // over the warp's valid tokens, then M - y in 16-bit fixed point
    {
        const int lane = t & 31, qw = t >> 5;
        float m_own[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            float w[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) w[r] = valid ? v[h][r] * a.scale2 : -INFINITY;
            m_own[h] = warp_rows_reduce<true>(w);
            if (h * 32 + lane < a.Rs)
                a.lmax[((static_cast<int64_t>(slab_local) * a.tiles_max + tile) * 4 + qw) * a.Rs + h * 32 + lane] =
                    m_own[h];
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(
            a.logits + (static_cast<int64_t>(slab_local) * a.rows_per_slab + tile * kTileTokens + t) * a.Rs);
#pragma unroll
        for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int r = 0; r < 32; r += 2) {
                const float M0 = __shfl_sync(0xffffffffu, m_own[h], r);
                const float M1 = __shfl_sync(0xffffffffu, m_own[h], r + 1);
                const uint32_t pk = quant_logit(M0, v[h][r] * a.scale2) | (quant_logit(M1, v[h][r + 1] * a.scale2) << 16);
                if (valid) dst[h * 16 + r / 2] = pk;
            }
    }
    const int64_t seg = static_cast<int64_t>(slab_local) * a.B + b;
    float2* out = a.rec + ((blockIdx.x + seg) * 2) * a.Rs;
    if (t < a.R) {
        out[a.Rs + t] = make_float2(-INFINITY, 0.0f);  // no second warpgroup here
        __threadfence();
    }
    stats_flush<NH>(rs, stats, t >> 5, 1, out, a.R);
    segment_done(a.tile_base, a.B, a.nslab, gridDim.x, seg, 2, a.rec, a.seg_cnt, a.lse2, a.R, a.Rs,
                 stats, &seg_flag, t >> 5, 1);
}

}  // namespace

cudaError_t launch_logits_simt(const Plan& pl, const sp_shape* s, const int32_t* seq_off,
                               const uint16_t* q, const uint16_t* k, void* ws, int slab0, int nslab,
                               int* grid_out, cudaStream_t st) {
    SimtArgs a;
    a.seq_off = seq_off;
    a.tile_base = ws_ptr<int32_t>(ws, pl.o_tile_base);
    a.q = q;
    a.k = k;
    a.logits = ws_ptr<uint16_t>(ws, pl.o_logits);
    a.lmax = ws_ptr<float>(ws, pl.o_lmax);
    a.tiles_max = pl.tiles_max;
    a.rec = ws_ptr<float2>(ws, pl.o_part);
    a.seg_cnt = ws_ptr<unsigned>(ws, pl.o_segcnt);
    a.lse2 = ws_ptr<float>(ws, pl.o_lse);
    a.bad = &ws_ptr<WsHeader>(ws, 0)->bad_input;
    a.B = pl.B;
    a.Hk = pl.Hk;
    a.G = pl.G;
    a.L = pl.L;
    a.R = pl.R;
    a.Rs = pl.Rs;
    a.d = pl.d;
    a.slab0 = slab0;
    a.nslab = nslab;
    a.rows_per_slab = pl.tiles_max * kTileTokens;
    a.ks_layer = s->k_stride_layer;
    a.ks_token = s->k_stride_token;
    a.ks_head = s->k_stride_head;
    a.qs_seq = s->q_stride_seq;
    a.qs_layer = s->q_stride_layer;
    a.qs_step = s->q_stride_step;
    a.qs_head = s->q_stride_head;
    a.scale2 = pl.scale2;
    const int grid = static_cast<int>(pl.tiles_max * nslab);
    *grid_out = grid;
    const int nh = pl.Rs > 32 ? 2 : 1;
    const size_t sm = static_cast<size_t>(32 * nh) * pl.d * sizeof(float);
    auto kern = nh == 2 ? logits_simt_kernel<2> : logits_simt_kernel<1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sm));
    if (e != cudaSuccess) return e;
    return launch_k(kern, grid, 128, sm, st, a);
}

}  // namespace sp

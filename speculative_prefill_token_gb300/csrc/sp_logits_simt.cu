// CUDA-core (FP32 FMA) variant of the logits kernel. Same contract and
// scratch layout as the tensor-core kernel: one CTA per (128-token tile,
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
    float* logits;
    float2* part;
    const int32_t* bad;
    int B, Hk, G, L, R, Rs, d, slab0;
    int64_t Ntot, tiles_max;
    int64_t ks_layer, ks_token, ks_head, qs_seq, qs_layer, qs_step, qs_head;
    float scale2;
};

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <int RMAX>
__global__ void __launch_bounds__(128) logits_simt_kernel(const SimtArgs a) {
    if (*a.bad) return;
    const int64_t tile = blockIdx.x;
    if (tile >= a.tile_base[a.B]) return;
    extern __shared__ float qs[];  // [RMAX][d]
    __shared__ float2 stats[4][RMAX];
    const int b = search_base(a.tile_base, a.B, tile);
    const int64_t i = tile - a.tile_base[b];
    const int64_t start = a.seq_off[b];
    const int64_t n = static_cast<int64_t>(a.seq_off[b + 1]) - start;
    const int64_t tok0 = start + i * kTileTokens;
    const int nvalid = static_cast<int>(min64(kTileTokens, n - i * kTileTokens));
    const int slab_local = blockIdx.y;
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
    float acc[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) acc[r] = 0.0f;
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
            for (int r = 0; r < RMAX; ++r) {
                const float* qr = qs + r * a.d + x0;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r] = fmaf(kf[e], qr[e], acc[r]);
            }
        }
    }
    float v[RMAX > 32 ? 2 : 1][32];
#pragma unroll
    for (int r = 0; r < (RMAX > 32 ? 64 : 32); ++r) {
        float x = (r < RMAX) ? acc[r < RMAX ? r : 0] : 0.0f;
        v[r >> 5][r & 31] = valid ? x * a.scale2 : -INFINITY;
    }
    if (valid) {
        float* dst = a.logits + (static_cast<int64_t>(slab_local) * a.Ntot + tok0 + t) * a.Rs;
        for (int r = 0; r < a.Rs; ++r) dst[r] = v[r >> 5][r & 31];
    }
    const int warp = t >> 5, lane = t & 31;
#pragma unroll
    for (int hh = 0; hh < (RMAX > 32 ? 2 : 1); ++hh) {
        const float2 pr = warp_row_partials(v[hh]);
        if (hh * 32 + lane < RMAX) stats[warp][hh * 32 + lane] = pr;
    }
    __syncthreads();
    if (t < a.R) {
        float2 acc2 = stats[0][t];
        acc2 = merge_partial(acc2, stats[1][t]);
        acc2 = merge_partial(acc2, stats[2][t]);
        acc2 = merge_partial(acc2, stats[3][t]);
        a.part[(static_cast<int64_t>(slab_local) * a.tiles_max + tile) * a.Rs + t] = acc2;
    }
}

}  // namespace

cudaError_t launch_logits_simt(const Plan& pl, const sp_shape* s, const int32_t* seq_off,
                               const uint16_t* q, const uint16_t* k, void* ws, int slab0, int nslab,
                               cudaStream_t st) {
    SimtArgs a;
    a.seq_off = seq_off;
    a.tile_base = ws_ptr<int32_t>(ws, pl.o_tile_base);
    a.q = q;
    a.k = k;
    a.logits = ws_ptr<float>(ws, pl.o_logits);
    a.part = ws_ptr<float2>(ws, pl.o_part);
    a.bad = &ws_ptr<WsHeader>(ws, 0)->bad_input;
    a.B = pl.B;
    a.Hk = pl.Hk;
    a.G = pl.G;
    a.L = pl.L;
    a.R = pl.R;
    a.Rs = pl.Rs;
    a.d = pl.d;
    a.slab0 = slab0;
    a.Ntot = pl.Ntot;
    a.tiles_max = pl.tiles_max;
    a.ks_layer = s->k_stride_layer;
    a.ks_token = s->k_stride_token;
    a.ks_head = s->k_stride_head;
    a.qs_seq = s->q_stride_seq;
    a.qs_layer = s->q_stride_layer;
    a.qs_step = s->q_stride_step;
    a.qs_head = s->q_stride_head;
    a.scale2 = pl.scale2;
    dim3 grid(static_cast<unsigned>(pl.tiles_max), static_cast<unsigned>(nslab));
    if (pl.R <= 8) {
        logits_simt_kernel<8><<<grid, 128, 8 * pl.d * sizeof(float), st>>>(a);
    } else if (pl.R <= 32) {
        logits_simt_kernel<32><<<grid, 128, 32 * pl.d * sizeof(float), st>>>(a);
    } else {
        const size_t sm = 64 * pl.d * sizeof(float);
        cudaFuncSetAttribute(logits_simt_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sm));
        logits_simt_kernel<64><<<grid, 128, sm, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace sp

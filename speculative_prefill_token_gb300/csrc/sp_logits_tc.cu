// Stand-alone logits kernel of the SpecPrefill scoring path (the logits
// phase of sp_logits_phase.cuh on its own), used by sp_attn_importance and
// the multi-wave path, and the host side of the phase: tensor maps, kernel
// arguments and shared-memory size.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_logits_phase.cuh"
#include "sp_ptx.cuh"

namespace sp {
namespace {

// Tile count of the call and, for small batches, this CTA's own tile
// offsets: the call's inputs (seq_off, Q, K) were complete before the prep
// kernel passed its own wait, so the producer and MMA warps start at once
// and only the epilogue waits for the prep kernel's counters; larger
// batches wait for the prep kernel's offsets. The kernel does not release
// its dependent early: the importance kernel then launches once this one
// has completed and spreads over every SM, instead of piling its CTAs onto
// the SMs this kernel frees first (2B workload 66.7 -> 65.8 us per call,
// 0.8B workload 39.4 -> 36.1 us).
// A single prompt with keys that are not block-paged takes its offsets from
// Ntot ({0, Ntot}; the prep kernel rejects anything else and the scores of
// such a call are never used), so the producer starts right after the
// setup; every key read stays inside the key map's Ntot rows.
__device__ __forceinline__ int64_t logits_start(const LogitsCtx& c, const TcArgs& a, PromptBounds pb,
                                                const int32_t** tb, const int32_t** so, int* epi_wait) {
    int64_t T;
    if (a.B <= kLocalPrompts) {
        int32_t* own = reinterpret_cast<int32_t*>(c.smem + c.L.tile_base);
        int32_t* own_so = own + kLocalPrompts + 1 + kThreads / 32;
        if (a.B == 1 && a.kv_mode != 2) {
            T = (a.Ntot + kTileTokens - 1) / kTileTokens;
            if (threadIdx.x == 0) {
                own[0] = 0;
                own[1] = static_cast<int32_t>(T);
                own_so[0] = 0;
                own_so[1] = static_cast<int32_t>(a.Ntot);
            }
            __syncthreads();
            if (T > a.tiles_max) T = a.tiles_max;
        } else {
            T = local_tile_base(a, pb, own);
        }
        *tb = own;
        *so = own_so;
        *epi_wait = 1;
    } else {
        grid_dep_wait();
        T = *a.bad ? 0 : a.tile_base[a.B];  // invalid offsets: no work, normal teardown
        *tb = a.tile_base;
        *so = a.seq_off;
        *epi_wait = 0;
    }
    return T;
}

template <int NH>
__global__ void __launch_bounds__(kThreads, 1)
    logits_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_s, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    LogitsCtx c = logits_ctx<NH>(smem_raw, a);
    const PromptBounds pb = logits_offsets_request(a);
    logits_setup(c, a, &tmap_k, &tmap_q, &tmap_s);
    const int32_t* tb;
    const int32_t* so;
    int epi_wait;
    const int64_t T = logits_start(c, a, pb, &tb, &so, &epi_wait);
    logits_phase<NH>(c, a, tb, so, epi_wait, &tmap_k, &tmap_q, &tmap_s, T, gridDim.x, blockIdx.x);
    logits_teardown(c, a);
}

// Per-layer key maps of a draft engine's cache (kv_mode 1 and 2), passed
// as one kernel parameter.
struct KvMaps {
    CUtensorMap m[kMaxKvLayers];
};

template <int NH>
__global__ void __launch_bounds__(kThreads, 1)
    logits_tc_kv_kernel(const __grid_constant__ KvMaps kmaps,
                        const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_s, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    LogitsCtx c = logits_ctx<NH>(smem_raw, a);
    const PromptBounds pb = logits_offsets_request(a);
    logits_setup(c, a, kmaps.m, &tmap_q, &tmap_s);
    const int32_t* tb;
    const int32_t* so;
    int epi_wait;
    const int64_t T = logits_start(c, a, pb, &tb, &so, &epi_wait);
    logits_phase<NH>(c, a, tb, so, epi_wait, kmaps.m, &tmap_q, &tmap_s, T, gridDim.x, blockIdx.x);
    logits_teardown(c, a);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}


}  // namespace

cudaError_t make_logits_maps(const Plan& pl, const sp_shape* s, const uint16_t* q, const uint16_t* k,
                             void* ws, int nslab, LogitsMaps* m) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int d = pl.d;
    {
        // K: dims (d, token, kv head, layer); unused strides get a harmless value
        const int64_t sh = pl.Hk > 1 ? s->k_stride_head : d;
        const int64_t sl = pl.Ly > 1 ? s->k_stride_layer : d;
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(pl.Ntot),
                              static_cast<cuuint64_t>(pl.Hk), static_cast<cuuint64_t>(pl.Ly)};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(s->k_stride_token) * 2,
                                 static_cast<cuuint64_t>(sh) * 2, static_cast<cuuint64_t>(sl) * 2};
        cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kTileTokens), 1, 1};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&m->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(k), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // Q: dims (d, q head, step, layer, prompt); box = the G heads x L steps of one slab
        const int64_t sh = pl.Hq > 1 ? s->q_stride_head : d;
        const int64_t ss = pl.L > 1 ? s->q_stride_step : d;
        const int64_t sl = pl.Ly > 1 ? s->q_stride_layer : d;
        const int64_t sb = pl.B > 1 ? s->q_stride_seq : d;
        cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(pl.Hq),
                              static_cast<cuuint64_t>(pl.L), static_cast<cuuint64_t>(pl.Ly),
                              static_cast<cuuint64_t>(pl.B)};
        cuuint64_t strides[4] = {static_cast<cuuint64_t>(sh) * 2, static_cast<cuuint64_t>(ss) * 2,
                                 static_cast<cuuint64_t>(sl) * 2, static_cast<cuuint64_t>(sb) * 2};
        cuuint32_t box[5] = {64, static_cast<cuuint32_t>(pl.G), static_cast<cuuint32_t>(pl.L), 1, 1};
        cuuint32_t es[5] = {1, 1, 1, 1, 1};
        if (enc(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<uint16_t*>(q), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // quantised logits scratch: dims (row value, tile slot row, slab); box = 32
        // values x 128 rows, staged as 64-byte rows with the 64-byte swizzle
        // (conflict-free staging stores; the global layout is dense)
        const uint64_t rows = static_cast<uint64_t>(pl.tiles_max) * kTileTokens;
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(pl.Rs), rows, static_cast<cuuint64_t>(nslab)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(pl.Rs) * 2,
                                 static_cast<cuuint64_t>(rows * pl.Rs * 2)};
        cuuint32_t box[3] = {32, static_cast<cuuint32_t>(kTileTokens), 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&m->s, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, ws_ptr<uint16_t>(ws, pl.o_logits), dims,
                strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

cudaError_t logits_smem(const Plan& pl, int* stages, uint32_t* smem, int* nh) {
    const int d_blocks = pl.d / 64;
    const uint32_t q_block_bytes = static_cast<uint32_t>(pl.Nmma) * 128u;
    *nh = pl.Rs > 32 ? 2 : 1;
    const uint32_t fixed = smem_layout(0, d_blocks, q_block_bytes, *nh).total + 1024;
    // A ring of kRingStages 16 KB stages (1.5 tiles in flight) already keeps the
    // key stream at its rate; the shared memory it leaves lets the small
    // kernels of other calls (streams) share the SM with a logits CTA.
    int st = static_cast<int>((kSmemLimit - static_cast<int>(fixed)) / kKBlockBytes);
    if (st > kRingStages) st = kRingStages;
    if (st < 2) return cudaErrorInvalidConfiguration;
    *stages = st;
    *smem = smem_layout(st, d_blocks, q_block_bytes, *nh).total + 1024;
    return cudaSuccess;
}

cudaError_t logits_config(const Plan& pl, const int32_t* seq_off, void* ws, int slab0, int nslab,
                          TcArgs* ap, uint32_t* smem, int* nh) {
    TcArgs& a = *ap;
    a.seq_off = seq_off;
    a.tile_base = ws_ptr<int32_t>(ws, pl.o_tile_base);
    a.lmax = ws_ptr<float>(ws, pl.o_lmax);
    a.tiles_max = pl.tiles_max;
    a.rec = ws_ptr<float2>(ws, pl.o_part);
    a.seg_cnt = ws_ptr<unsigned>(ws, pl.o_segcnt);
    a.lse2 = ws_ptr<float>(ws, pl.o_lse);
    a.status = &ws_ptr<WsHeader>(ws, 0)->status;
    a.bad = &ws_ptr<WsHeader>(ws, 0)->bad_input;
    a.B = pl.B;
    a.Hk = pl.Hk;
    a.G = pl.G;
    a.R = pl.R;
    a.Rs = pl.Rs;
    a.d_blocks = pl.d / 64;
    a.Nmma = pl.Nmma;
    a.Nacc = pl.Nacc;
    a.slab0 = slab0;
    a.nslab = nslab;
    a.q_block_bytes = static_cast<uint32_t>(pl.Nmma) * 128u;
    a.scale2 = pl.scale2;
    a.spin = pl.spin;
    a.kv_mode = 0;
    a.Ntot = pl.Ntot;
    a.n_layers = pl.Ly;
    a.block_table = nullptr;
    a.block_size = 0;
    a.table_stride = 0;
    a.box_h = kTileTokens;
    a.nbox = 1;
    a.pool_tokens = pl.Ntot;
    return logits_smem(pl, &a.stages, smem, nh);
}

namespace {

// Tokens per K box of a key source: one 128-token box, or one box per block
// of a block-paged cache whose blocks are shorter than a tile.
int kv_box_h(const KvSrc* kv) {
    return (kv && kv->block_table && kv->block_size < kTileTokens) ? kv->block_size : kTileTokens;
}

cudaError_t make_kv_maps(const Plan& pl, const sp_shape* s, const KvSrc* kv, KvMaps* km) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int d = pl.d;
    const int64_t sh = pl.Hk > 1 ? s->k_stride_head : d;
    for (int l = 0; l < pl.Ly; ++l) {
        // dims (d, pool row, kv head, 1)
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(kv->pool_tokens),
                              static_cast<cuuint64_t>(pl.Hk), 1};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(s->k_stride_token) * 2,
                                 static_cast<cuuint64_t>(sh) * 2,
                                 static_cast<cuuint64_t>(s->k_stride_token) * 2 *
                                     static_cast<cuuint64_t>(kv->pool_tokens)};
        cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kv_box_h(kv)), 1, 1};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&km->m[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(kv->layer_k[l]),
                dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

}  // namespace

int logits_tc_grid(const Plan& pl, int nslab) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t work = pl.tiles_max * nslab;
    return static_cast<int>(work < sms ? work : sms);
}

cudaError_t launch_logits_tc(const Plan& pl, const sp_shape* s, const int32_t* seq_off,
                             const uint16_t* q, const uint16_t* k, void* ws, int slab0, int nslab,
                             int grid, cudaStream_t st, const KvSrc* kv) {
    LogitsMaps m;
    // without a key source the single K map addresses k; with one, the
    // single map is not used (it is built over the first layer's pool)
    cudaError_t err = make_logits_maps(pl, s, q, kv ? kv->layer_k[0] : k, ws, nslab, &m);
    if (err != cudaSuccess) return err;
    TcArgs a;
    uint32_t smem = 0;
    int nh = 1;
    if ((err = logits_config(pl, seq_off, ws, slab0, nslab, &a, &smem, &nh)) != cudaSuccess) return err;
    if (!kv) {
        auto kern = nh == 2 ? logits_tc_kernel<2> : logits_tc_kernel<1>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        return launch_k(kern, grid, kThreads, smem, st, m.k, m.q, m.s, a);
    }
    KvMaps km;  // the launch copies the maps into the kernel's parameter space
    if ((err = make_kv_maps(pl, s, kv, &km)) != cudaSuccess) return err;
    a.kv_mode = kv->block_table ? 2 : 1;
    a.n_layers = pl.Ly;
    a.block_table = kv->block_table;
    a.block_size = kv->block_table ? kv->block_size : 0;
    a.table_stride = kv->table_stride;
    a.box_h = kv_box_h(kv);
    a.nbox = kTileTokens / a.box_h;
    a.pool_tokens = kv->pool_tokens;
    auto kern = nh == 2 ? logits_tc_kv_kernel<2> : logits_tc_kv_kernel<1>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_k(kern, grid, kThreads, smem, st, km, m.q, m.s, a);
}

}  // namespace sp

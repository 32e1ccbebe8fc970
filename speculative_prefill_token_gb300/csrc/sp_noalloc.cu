// Allocation-free variant of the pool + chunk-score stage.
//
// Some callers cannot hand the library a workspace: they run where device
// memory may not be allocated after start-up (a serving loop that owns all
// device memory through its own pool and forbids further allocations, or a
// plugin whose host runtime exposes no allocator to it), or where a
// cudaMalloc/cudaFree would be too costly because either call can
// synchronise the device. For them this entry point keeps its scratch in a
// fixed array that is part of the library's device image, so a call
// allocates nothing. The caller still passes every input and output.
//
// The array is created once per GPU when the library's device code is
// loaded on that GPU and lives until the process exits. Every call on a GPU
// uses the same array, so calls that overlap on the GPU (different streams,
// or different host threads, without ordering between them) race on it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sp_internal.h"
#include "specprefill.h"

namespace sp {
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB on every GPU
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_pool_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_pool_scratch on the current GPU, looked up once per
// GPU (the symbol's host-side name is not a device address).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_pool_scratch);
        if (e != cudaSuccess || p == nullptr) return SP_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SP_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace sp

using namespace sp;

extern "C" int sp_pool_chunk_noalloc(const sp_shape* shape, const sp_params* params,
                                     const int32_t* seq_off, const float* imp, float* tok_score,
                                     float* chunk_score, int32_t* chunk_off, int32_t* status_out,
                                     sp_stream_t stream) {
    Plan pl;
    int rc = make_plan(shape, params, &pl);
    if (rc != SP_OK) return rc;
    if (!seq_off || !imp || !tok_score || !chunk_score || !chunk_off) return SP_ERR_INVALID_ARG;
    // scratch layout inside the fixed array: header, the four offset tables
    // and the counters the prep kernel writes, per-block (min, max) of the
    // pooled scores
    size_t off = sizeof(WsHeader);
    const size_t tables = (static_cast<size_t>(pl.B) + 1) * sizeof(int32_t);
    pl.o_tile_base = off;
    off = align256(off + tables);
    pl.o_chunk_off = off;
    off = align256(off + tables);
    pl.o_pblk_base = off;
    off = align256(off + tables);
    pl.o_slice_base = off;
    off = align256(off + tables);
    pl.o_segcnt = off;
    pl.o_lcount = off + static_cast<size_t>(pl.slabs_per_wave) * pl.B * sizeof(int32_t);
    off = align256(off + (static_cast<size_t>(pl.slabs_per_wave) + 1) * pl.B * sizeof(int32_t));
    pl.o_ppart = off;
    off = align256(off + static_cast<size_t>(pl.pblk_max) * 2 * sizeof(float));
    if (off > kStaticScratchBytes) return SP_ERR_UNSUPPORTED;  // batch too large for the fixed scratch
    void* ws = nullptr;
    if ((rc = scratch_address(&ws)) != SP_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the previous call's status word, input flag and counter must not leak in
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return SP_ERR_CUDA;
    if (launch_prep(pl, seq_off, ws, chunk_off, st) != cudaSuccess) return SP_ERR_CUDA;
    const sp_params pp = post_params(params);
    if (launch_pool(pl, &pp, seq_off, imp, tok_score, ws, st) != cudaSuccess) return SP_ERR_CUDA;
    if (launch_chunk(pl, &pp, seq_off, tok_score, chunk_score, ws, st) != cudaSuccess)
        return SP_ERR_CUDA;
    if (status_out &&
        cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return SP_ERR_CUDA;
    return SP_OK;
}

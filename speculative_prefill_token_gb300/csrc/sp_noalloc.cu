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
// The array is created once per CUDA context when the library's device
// code is loaded into that context (normally once per GPU, the primary
// context) and lives until the context is destroyed (process exit, or a
// cudaDeviceReset, after which a new context gets a new copy). Every call in
// a context uses the same array, so calls that overlap on the GPU
// (different streams, or different host threads, without ordering between
// them) race on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sp_internal.h"
#include "specprefill.h"

namespace sp {
namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB per context
constexpr int kMaxContexts = 64;

static __device__ __align__(256) unsigned char g_pool_scratch[kStaticScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

std::mutex g_mutex;
CUcontext g_ctx[kMaxContexts] = {};
void* g_addr[kMaxContexts] = {};
int g_next = 0;

// Device address of g_pool_scratch in the calling thread's current context
// (the symbol's host-side name is not a device address). Outside stream
// capture it is looked up on every call, so a context created after a
// cudaDeviceReset (whose module, and array, may sit elsewhere) is never
// given a stale address; during capture the last address found for the
// same context is reused, because the lookup may load the module, which a
// capture does not allow.
int scratch_address(cudaStream_t st, void** out) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return SP_ERR_CUDA;
    void* p = nullptr;
    if (cap == cudaStreamCaptureStatusNone) {
        // also makes the device's primary context current for this thread
        const cudaError_t e = cudaGetSymbolAddress(&p, g_pool_scratch);
        if (e != cudaSuccess || p == nullptr) return SP_ERR_CUDA;
    }
    CtxGetCurrentFn get = ctx_fn();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    int slot = -1;
    for (int i = 0; i < kMaxContexts; ++i)
        if (g_ctx[i] == ctx) slot = i;
    if (cap == cudaStreamCaptureStatusNone) {
        if (slot < 0) {
            slot = g_next;
            g_next = (g_next + 1) % kMaxContexts;
            g_ctx[slot] = ctx;
        }
        g_addr[slot] = p;
    } else if (slot < 0) {
        return SP_ERR_UNSUPPORTED;  // no uncaptured call in this context yet
    }
    *out = g_addr[slot];
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
    // the prep kernel writes, per-block (min, max) of the pooled scores; the
    // prep kernel's per-segment counters are not needed by pool and chunk and
    // get no room (it is told to zero none)
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
    pl.o_lcount = off;
    pl.o_ppart = off;
    off = align256(off + static_cast<size_t>(pl.pblk_max) * 2 * sizeof(float));
    if (off > kStaticScratchBytes) return SP_ERR_UNSUPPORTED;  // batch too large for the fixed scratch
    void* ws = nullptr;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((rc = scratch_address(st, &ws)) != SP_OK) return rc;
    // the previous call's status word, input flag and counter must not leak in
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return SP_ERR_CUDA;
    if (launch_prep(pl, seq_off, ws, chunk_off, st, 0) != cudaSuccess) return SP_ERR_CUDA;
    const sp_params pp = post_params(params);
    if (launch_pool(pl, &pp, seq_off, imp, tok_score, ws, st) != cudaSuccess) return SP_ERR_CUDA;
    if (launch_chunk(pl, &pp, seq_off, tok_score, chunk_score, ws, st) != cudaSuccess)
        return SP_ERR_CUDA;
    if (status_out &&
        cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return SP_ERR_CUDA;
    return SP_OK;
}

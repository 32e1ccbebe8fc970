// The logits phase of the SpecPrefill scoring path on fifth-generation
// tensor cores (sm_103a), shared by the logits kernels for dense and for
// in-situ (per-layer, block-paged) key sources.
//
// For one (layer l, KV head g) "slab" and one prompt, the logits are
//   s[t, r] = <k[l, t, g, :], q[l, step(r), g*G + head(r), :]>   (unscaled)
// for the prompt's tokens t and the R = L*G query rows r = step*G + head
// sharing KV head g ("SpecPrefill — Implementation Guide", §How It Works /
// Attention Capture and Token Importance: one post-softmax row per head and
// lookahead step; the attention matrix is Q K^T, §Sliding Window / The OOM
// Problem). Only R rows per slab are needed, so this is a tall-skinny GEMM
// that streams every key exactly once from HBM:
//   A = 128 keys x 64 head-dim elements (one TMA box, 128-byte swizzle),
//   B = R query rows x 64 elements, D = 128 x N fp32 in tensor memory.
//
// Roles (320 threads, one CTA per SM, persistent over a contiguous range of
// (slab, prompt, 128-token tile) work items):
//   warp 8      TMA producer: K boxes into a ring of 16 KB stages, Q per
//               (slab, prompt) into one of two buffers;
//   warp 9      tcgen05.mma issuer (one thread) and TMEM owner;
//   warps 0-7   two epilogue warpgroups; warpgroup e drains TMEM accumulator
//               e (tiles alternate). Per tile, each warp (32 tokens) takes
//               the row maxima M of the scaled logits (butterfly), stages the
//               tile's logits as 16-bit M - y in shared memory for one TMA
//               store into the scratch (one 128-token slot per tile), and
//               sums exp2(y - M) per row (butterfly); lane r merges the pair
//               into its running softmax statistics of row r. Once per (slab,
//               prompt) segment the four warps' pairs are merged into a
//               record; the last contribution to a segment merges its
//               records into the segment's log2 normaliser.
// Every mbarrier wait is bounded; a wait that gives up records
// SP_ERR_TIMEOUT in the workspace status word, and the CTA then drains its
// own copies, stores and MMAs in flight before it leaves the phase.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_ptx.cuh"

namespace sp {


constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kKBlockBytes = kTileTokens * 128;  // 128 tokens x 64 bf16
constexpr int kStageOutBytes = kTileTokens * 64;   // 128 tokens x 32 quantised 16-bit logits
constexpr int kMaxStages = 16;
constexpr int kRingStages = 6;   // stages the host configures (at most kMaxStages)
constexpr int kAcc = 4;                          // TMEM accumulators (tiles in flight)
constexpr int kSmemLimit = 232448;              // per-block opt-in maximum on sm_100-class parts
constexpr int64_t kDrainSpin = int64_t(1) << 22;

struct TcArgs {
    const int32_t* seq_off;
    const int32_t* tile_base;
    float* lmax;     // per (slab, tile, warp quarter) row maxima of the scaled logits [..][Rs]
    int64_t tiles_max;
    float2* rec;     // per (CTA, segment, warpgroup) softmax records [.. * 2 + wg][Rs]
    unsigned* seg_cnt;  // per segment: records written so far (zero between calls)
    float* lse2;     // per segment normaliser [seg][Rs]
    int32_t* status;
    const int32_t* bad;
    int B, Hk, G, R, Rs, d_blocks, Nmma, Nacc, slab0, nslab, stages;
    uint32_t q_block_bytes;  // Nmma * 128
    float scale2;
    int64_t spin;
    // key source: 0 = one tensor map (token, head, layer); 1 = one map per
    // layer, packed token index; 2 = one map per layer, block-paged
    int kv_mode, n_layers;
    int64_t Ntot;
    const int32_t* block_table;  // kv_mode 2: [B][table_stride]
    int block_size, table_stride, box_h, nbox;  // box_h tokens per TMA box, nbox boxes per tile
    int64_t pool_tokens;
};

struct SmemLayout {
    uint32_t k_ring, q_buf, out_buf, bars, tmem_slot, abort_flag, seg_flag, stats, tile_base, total;
};

// Batches of at most this many prompts get their tile offsets computed by
// every CTA of the logits kernel itself (from seq_off, a call input), so
// that its producer and MMA warps need not wait for the prep kernel.
constexpr int kLocalPrompts = 256;

__host__ __device__ inline SmemLayout smem_layout(int stages, int d_blocks, uint32_t q_block_bytes,
                                                  int nh) {
    SmemLayout s;
    uint32_t off = 0;
    s.k_ring = off;
    off += static_cast<uint32_t>(stages) * kKBlockBytes;
    s.q_buf = off;
    off += 2u * static_cast<uint32_t>(d_blocks) * q_block_bytes;
    off = (off + 1023u) & ~1023u;
    s.out_buf = off;                                   // [warpgroup][half] 16 KB, swizzled
    off += 2u * static_cast<uint32_t>(nh) * kStageOutBytes;
    s.bars = off;
    off += 8u * (2 * kMaxStages + 13);
    s.tmem_slot = off;
    off += 8;
    s.abort_flag = off;
    off += 8;
    s.seg_flag = off;  // [warpgroup] int
    off += 8;
    s.stats = off;
    off += 2u * 4u * 64u * 8u;  // [warpgroup][warp][row] float2
    s.tile_base = off;          // [kLocalPrompts + 1] int32, per-warp sums, then seq_off
    off += 4u * (2 * (kLocalPrompts + 1) + kThreads / 32);
    s.total = off;
    return s;
}

struct Item {
    int slab;    // local slab index in [0, nslab)
    int b;       // prompt
    int tile;    // flattened tile index of the slab (scratch slot)
    int tok0;    // first global token of the tile (token counts fit 31 bits)
    int nvalid;  // tokens of the tile inside the prompt
};

// Walks a CTA's contiguous range of work items. Consecutive items are
// consecutive tiles of one prompt except at prompt and slab boundaries, so
// only those re-read the offsets; every other step is arithmetic.
struct ItemCursor {
    Item it;
    int base_b;  // first tile of the current prompt
    int next_b;  // first tile of the next prompt
    int start, n;

    const int32_t* tb;  // the batch's tile offsets (the CTA's own copy or the prep kernel's)
    const int32_t* so;  // the batch's token offsets (the CTA's own copy or seq_off)

    __device__ __forceinline__ void set(const TcArgs& a, int64_t w, int64_t T) {
        it.slab = static_cast<int>(w / T);
        it.tile = static_cast<int>(w - static_cast<int64_t>(it.slab) * T);
        it.b = search_base(tb, a.B, it.tile);
        base_b = tb[it.b];
        next_b = tb[it.b + 1];
        start = so[it.b];
        n = so[it.b + 1] - start;
        place();
    }
    __device__ __forceinline__ void place() {
        const int i = it.tile - base_b;
        it.tok0 = start + i * kTileTokens;
        const int rem = n - i * kTileTokens;
        it.nvalid = rem < kTileTokens ? rem : kTileTokens;
    }
    // Moves to item w, the successor of the current one.
    __device__ __forceinline__ void next(const TcArgs& a, int64_t w, int64_t T) {
        const int tile = it.tile + 1;
        if (tile < next_b && tile < T) {
            it.tile = tile;
            place();
        } else {
            set(a, w, T);
        }
    }
};

__device__ __forceinline__ void record_timeout(const TcArgs& a, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicCAS(a.status, 0, static_cast<int32_t>(SP_ERR_TIMEOUT));
}


// Shared-memory addresses of one CTA of the logits phase.
struct LogitsCtx {
    uint8_t* smem;
    SmemLayout L;
    uint32_t base, k_ring, q_buf, bar_full, bar_empty, bar_qfull, bar_qempty, bar_tfull, bar_tempty,
        bar_drain, q_stage_bytes, tmem_base;
    volatile uint32_t* tmem_slot;
    volatile int* abort_flag;
    float2* stats;
};

template <int NH>
__device__ __forceinline__ LogitsCtx logits_ctx(uint8_t* smem_raw, const TcArgs& a) {
    LogitsCtx c;
    c.smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~static_cast<uintptr_t>(1023));
    c.L = smem_layout(a.stages, a.d_blocks, a.q_block_bytes, NH);
    c.base = smem_u32(c.smem);
    c.k_ring = c.base + c.L.k_ring;
    c.q_buf = c.base + c.L.q_buf;
    c.bar_full = c.base + c.L.bars;
    c.bar_empty = c.bar_full + 8 * kMaxStages;
    c.bar_qfull = c.bar_empty + 8 * kMaxStages;   // [2]
    c.bar_qempty = c.bar_qfull + 16;              // [2]
    c.bar_tfull = c.bar_qempty + 16;              // [4]
    c.bar_tempty = c.bar_tfull + 32;              // [4]
    c.bar_drain = c.bar_tempty + 32;              // [1]
    c.tmem_slot = reinterpret_cast<volatile uint32_t*>(c.smem + c.L.tmem_slot);
    c.abort_flag = reinterpret_cast<volatile int*>(c.smem + c.L.abort_flag);
    c.stats = reinterpret_cast<float2*>(c.smem + c.L.stats);
    c.q_stage_bytes = static_cast<uint32_t>(a.d_blocks) * a.q_block_bytes;
    c.tmem_base = 0;
    return c;
}

// Initialise the phase's mbarriers and abort flag (thread 0; the caller
// synchronises the CTA before any thread uses them).
__device__ __forceinline__ void logits_init_barriers(const LogitsCtx& c, const TcArgs& a) {
    for (int s = 0; s < a.stages; ++s) {
        mbar_init(c.bar_full + 8 * s, 1);
        mbar_init(c.bar_empty + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
        mbar_init(c.bar_qfull + 8 * i, 1);
        mbar_init(c.bar_qempty + 8 * i, 1);
    }
    for (int i = 0; i < kAcc; ++i) {
        mbar_init(c.bar_tfull + 8 * i, 1);
        mbar_init(c.bar_tempty + 8 * i, 128);
    }
    mbar_init(c.bar_drain, 1);
    *c.abort_flag = 0;
    fence_mbar_init();
}

// Setup by all kThreads threads, touching only this CTA's shared and tensor
// memory: barriers, zeroed Q buffers (rows >= R stay zero), TMEM.
__device__ __forceinline__ void logits_setup(LogitsCtx& c, const TcArgs& a, const CUtensorMap* tmap_k,
                                             const CUtensorMap* tmap_q, const CUtensorMap* tmap_s) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) logits_init_barriers(c, a);
    {
        uint4* qz = reinterpret_cast<uint4*>(c.smem + c.L.q_buf);
        const int n16 = static_cast<int>(2 * c.q_stage_bytes / 16);
        for (int i = threadIdx.x; i < n16; i += kThreads) qz[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(c.tmem_slot)), static_cast<uint32_t>(kAcc * a.Nacc));
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        for (int l = 0; l < (a.kv_mode ? a.n_layers : 1); ++l) prefetch_tmap(tmap_k + l);
        prefetch_tmap(tmap_q);
        prefetch_tmap(tmap_s);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem_base = *c.tmem_slot;
}

// Tile offsets of the batch computed by this CTA (all kThreads threads,
// B <= kLocalPrompts) from seq_off: tb[b] = sum over earlier prompts of
// ceil(n / 128), tb[B] the total, and a copy of seq_off after the per-warp
// sums (tb + kLocalPrompts + 1 + kThreads / 32); returns the tile count, 0
// when seq_off is not a valid packing of Ntot tokens (or, for a block-paged
// key source, a prompt has more blocks than its table row), as the prep
// kernel decides.
// The prompt bounds of thread t < B, requested (by logits_offsets_request)
// before the CTA's setup so that their latency overlaps it.
struct PromptBounds {
    int32_t lo, hi;
};

__device__ __forceinline__ PromptBounds logits_offsets_request(const TcArgs& a) {
    PromptBounds pb{0, 0};
    const int t = threadIdx.x;
    // (a single unpaged prompt takes its bounds from Ntot: see logits_start)
    if (a.B <= kLocalPrompts && t < a.B && !(a.B == 1 && a.kv_mode != 2)) {
        pb.lo = a.seq_off[t];
        pb.hi = a.seq_off[t + 1];
    }
    return pb;
}

__device__ __forceinline__ int64_t local_tile_base(const TcArgs& a, PromptBounds pb, int32_t* tb) {
    int32_t* warp_sum = tb + kLocalPrompts + 1;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int ok = 1;
    int32_t tiles = 0;
    if (t < a.B) {
        const int64_t n = static_cast<int64_t>(pb.hi) - pb.lo;
        if (n < 0) ok = 0;
        if (a.kv_mode == 2 && (n + a.block_size - 1) / a.block_size > a.table_stride) ok = 0;
        tiles = n > 0 ? static_cast<int32_t>((n + kTileTokens - 1) / kTileTokens) : 0;
        if (t == 0 && pb.lo != 0) ok = 0;
        if (t == a.B - 1 && static_cast<int64_t>(pb.hi) != a.Ntot) ok = 0;
    }
    int32_t incl = tiles;
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    ok = __syncthreads_and(ok);
    int32_t before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    int32_t* so = warp_sum + kThreads / 32;  // the CTA's copy of seq_off
    if (t < a.B) {
        tb[t] = before + incl - tiles;
        so[t] = pb.lo;
    }
    if (t == a.B - 1) {
        tb[a.B] = before + incl;
        so[a.B] = pb.hi;
    }
    __syncthreads();
    const int64_t T = ok ? static_cast<int64_t>(tb[a.B]) : 0;
    return T < a.tiles_max ? T : a.tiles_max;
}

// Frees the tensor memory (all kThreads threads).
__device__ __forceinline__ void logits_teardown(const LogitsCtx& c, const TcArgs& a) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(c.tmem_base, static_cast<uint32_t>(kAcc * a.Nacc));
    }
}

// Block-paged keys (kv_mode 2). Box j of a tile covers logical tokens
// [t, t + box_h) of the prompt, t = 128 i + j box_h, inside one block;
// boxes past the prompt's end read its last block (those rows are masked
// later). paged_block requests the block id of box `lane` of the cursor's
// tile without using it (so the lane does not wait for it); paged_row turns
// it into a key-map row when the copies are issued, and reports a block
// outside the pool (replaced by row 0).
__device__ __forceinline__ int paged_block(const TcArgs& a, const ItemCursor& cur, int lane) {
    if (lane >= a.nbox) return 0;
    const int64_t t = static_cast<int64_t>(cur.it.tile - cur.base_b) * kTileTokens +
                      static_cast<int64_t>(lane) * a.box_h;
    const int64_t lb = min64(t / a.block_size, (static_cast<int64_t>(cur.n) - 1) / a.block_size);
    return a.block_table[static_cast<int64_t>(cur.it.b) * a.table_stride + lb];
}

__device__ __forceinline__ int paged_row(const TcArgs& a, const ItemCursor& cur, int lane, int page) {
    if (lane >= a.nbox) return 0;
    const int64_t t = static_cast<int64_t>(cur.it.tile - cur.base_b) * kTileTokens +
                      static_cast<int64_t>(lane) * a.box_h;
    const int64_t row = static_cast<int64_t>(page) * a.block_size + t % a.block_size;
    if (page < 0 || row + a.box_h > a.pool_tokens) {
        atomicCAS(a.status, 0, static_cast<int32_t>(SP_ERR_DEVICE));
        return 0;
    }
    return static_cast<int>(row);
}

// Producer of the block-paged path, run by the whole producer warp: lane 0
// waits on the ring, lane j issues box j of each 16 KB stage (nbox boxes);
// lane j < nbox looks up the block of box j three items ahead, so that
// the table's latency overlaps the copies of the items before it (also at
// the start, where the ring is still empty).
__device__ __forceinline__ void produce_paged(const LogitsCtx& c, const TcArgs& a, const int32_t* tb,
                                              const int32_t* so, const CUtensorMap* tmap_k, const CUtensorMap* tmap_q,
                                              int64_t T, int64_t w_begin, int64_t w_end, int lane) {
    constexpr unsigned kFull = 0xffffffffu;
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    int qn = 0;
    int64_t prev_key = -1;
    uint32_t issued_phase[kMaxStages];
    bool issued[kMaxStages];
    for (int s = 0; s < kMaxStages; ++s) issued[s] = false;
    bool ok = true;
    // block ids of the current item (p0) and of the next three (p1..p3);
    // `ahead` is the cursor of the last item looked up
    ItemCursor cur, ahead;
    cur.tb = tb;
    cur.so = so;
    int p0 = 0, p1 = 0, p2 = 0, p3 = 0;
    if (w_begin < w_end) {
        cur.set(a, w_begin, T);
        ahead = cur;
        p0 = paged_block(a, ahead, lane);
        if (w_begin + 1 < w_end) {
            ahead.next(a, w_begin + 1, T);
            p1 = paged_block(a, ahead, lane);
        }
        if (w_begin + 2 < w_end) {
            ahead.next(a, w_begin + 2, T);
            p2 = paged_block(a, ahead, lane);
        }
        if (w_begin + 3 < w_end) {
            ahead.next(a, w_begin + 3, T);
            p3 = paged_block(a, ahead, lane);
        }
    }
    for (int64_t w = w_begin; w < w_end; ++w) {
        if (w > w_begin) cur.next(a, w, T);
        const int row = paged_row(a, cur, lane, p0);
        int pn = 0;
        if (w + 4 < w_end) {
            ahead.next(a, w + 4, T);
            pn = paged_block(a, ahead, lane);
        }
        const Item& it = cur.it;
        const int slab = a.slab0 + it.slab;
        const int layer = slab / a.Hk, g = slab - layer * a.Hk;
        const int64_t key = static_cast<int64_t>(it.slab) * a.B + it.b;
        if (key != prev_key) {
            const int qb = qn & 1;
            if (lane == 0 && !mbar_wait_bounded(c.bar_qempty + 8 * qb, ((qn >> 1) & 1) ^ 1, a.spin,
                                                c.abort_flag)) {
                record_timeout(a, c.abort_flag);
                ok = false;
            }
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(c.bar_qfull + 8 * qb, static_cast<uint32_t>(a.R) * 128u * a.d_blocks);
                for (int kb = 0; kb < a.d_blocks; ++kb)
                    tma_load_5d(c.q_buf + qb * c.q_stage_bytes + kb * a.q_block_bytes, tmap_q,
                                c.bar_qfull + 8 * qb, kb * 64, g * a.G, 0, layer, it.b);
            }
            ++qn;
            prev_key = key;
        }
        for (int kb = 0; kb < a.d_blocks; ++kb) {
            if (lane == 0 && !mbar_wait_bounded(c.bar_empty + 8 * stage, phase ^ 1, a.spin, c.abort_flag)) {
                record_timeout(a, c.abort_flag);
                ok = false;
            }
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(c.bar_full + 8 * stage, kKBlockBytes);
            __syncwarp();
            // lane j issues box j of the stage (its own block's row): one
            // thread issuing all of a stage's boxes set the rate of small blocks
            if (lane < a.nbox)
                tma_load_4d(c.k_ring + stage * kKBlockBytes + static_cast<uint32_t>(lane * a.box_h) * 128u,
                            tmap_k + layer, c.bar_full + 8 * stage, kb * 64, row, g, 0, pol);
            if (lane == 0) {
                issued[stage] = true;
                issued_phase[stage] = phase;
            }
            if (++stage == a.stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (!ok) break;
        p0 = p1;
        p1 = p2;
        p2 = p3;
        p3 = pn;
    }
    if (lane == 0) {
        // drain: every copy this thread issued must land before exit
        for (int s = 0; s < a.stages; ++s)
            if (issued[s]) mbar_wait_spin(c.bar_full + 8 * s, issued_phase[s], kDrainSpin);
        for (int i = 0; i < 2 && i < qn; ++i) {
            const int last = (qn - 1 - i);
            mbar_wait_spin(c.bar_qfull + 8 * (last & 1), (last >> 1) & 1, kDrainSpin);
        }
    }
}

// The work of CTA `cta` of C over the T tiles of each of the wave's slabs.
// On return every TMA store of this CTA has completed; the CTA is not
// synchronised.
template <int NH>
__device__ __forceinline__ void logits_phase(const LogitsCtx& c, const TcArgs& a, const int32_t* tb,
                                             const int32_t* so, int epi_wait,
                                             const CUtensorMap* tmap_k,
                                             const CUtensorMap* tmap_q, const CUtensorMap* tmap_s,
                                             int64_t T, int64_t C, int64_t cta) {
    uint8_t* const smem = c.smem;
    const SmemLayout& L = c.L;
    const uint32_t k_ring = c.k_ring, q_buf = c.q_buf, bar_full = c.bar_full, bar_empty = c.bar_empty,
                   bar_qfull = c.bar_qfull, bar_qempty = c.bar_qempty, bar_tfull = c.bar_tfull,
                   bar_tempty = c.bar_tempty, bar_drain = c.bar_drain, q_stage_bytes = c.q_stage_bytes,
                   tmem_base = c.tmem_base;
    volatile int* abort_flag = c.abort_flag;
    float2* stats = c.stats;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t W = T * a.nslab;
    const int64_t w_begin = split_start(W, C, cta);
    const int64_t w_end = split_start(W, C, cta + 1);

    if (warp == kProducerWarp && a.kv_mode == 2) {
        produce_paged(c, a, tb, so, tmap_k, tmap_q, T, w_begin, w_end, lane);
    } else if (warp == kProducerWarp) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            int qn = 0;
            int64_t prev_key = -1;
            uint32_t issued_phase[kMaxStages];
            bool issued[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) issued[s] = false;
            bool ok = true;
            ItemCursor cur;
            cur.tb = tb;
            cur.so = so;
            for (int64_t w = w_begin; w < w_end && ok; ++w) {
                if (w == w_begin) cur.set(a, w, T);
                else cur.next(a, w, T);
                const Item& it = cur.it;
                const int slab = a.slab0 + it.slab;
                const int layer = slab / a.Hk, g = slab - layer * a.Hk;
                const int64_t key = static_cast<int64_t>(it.slab) * a.B + it.b;
                if (key != prev_key) {
                    const int qb = qn & 1;
                    if (!mbar_wait_bounded(bar_qempty + 8 * qb, ((qn >> 1) & 1) ^ 1, a.spin, abort_flag)) {
                        record_timeout(a, abort_flag);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar_qfull + 8 * qb,
                                          static_cast<uint32_t>(a.R) * 128u * a.d_blocks);
                    for (int kb = 0; kb < a.d_blocks; ++kb)
                        tma_load_5d(q_buf + qb * q_stage_bytes + kb * a.q_block_bytes, tmap_q,
                                    bar_qfull + 8 * qb, kb * 64, g * a.G, 0, layer, it.b);
                    ++qn;
                    prev_key = key;
                }
                for (int kb = 0; kb < a.d_blocks; ++kb) {
                    if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1, a.spin, abort_flag)) {
                        record_timeout(a, abort_flag);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar_full + 8 * stage, kKBlockBytes);
                    tma_load_4d(k_ring + stage * kKBlockBytes, a.kv_mode ? tmap_k + layer : tmap_k,
                                bar_full + 8 * stage, kb * 64, it.tok0, g, a.kv_mode ? 0 : layer, pol);
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == a.stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // drain: every copy this thread issued must land before exit
            for (int s = 0; s < a.stages; ++s)
                if (issued[s]) mbar_wait_spin(bar_full + 8 * s, issued_phase[s], kDrainSpin);
            for (int i = 0; i < 2 && i < qn; ++i) {
                const int last = (qn - 1 - i);
                mbar_wait_spin(bar_qfull + 8 * (last & 1), (last >> 1) & 1, kDrainSpin);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, a.Nmma);
            int stage = 0;
            uint32_t phase = 0;
            int qn = 0;
            int64_t prev_key = -1;
            int64_t j = 0;
            int qb = 0;
            bool ok = true;
            bool any_mma = false;
            ItemCursor cur;
            cur.tb = tb;
            cur.so = so;
            for (int64_t w = w_begin; w < w_end && ok; ++w, ++j) {
                if (w == w_begin) cur.set(a, w, T);
                else cur.next(a, w, T);
                const Item& it = cur.it;
                const int64_t key = static_cast<int64_t>(it.slab) * a.B + it.b;
                if (key != prev_key) {
                    if (qn > 0) tc_commit(bar_qempty + 8 * ((qn - 1) & 1));
                    qb = qn & 1;
                    if (!mbar_wait_bounded(bar_qfull + 8 * qb, (qn >> 1) & 1, a.spin, abort_flag)) {
                        record_timeout(a, abort_flag);
                        ok = false;
                        break;
                    }
                    ++qn;
                    prev_key = key;
                }
                const int acc = static_cast<int>(j & (kAcc - 1));
                if (!mbar_wait_bounded(bar_tempty + 8 * acc, static_cast<uint32_t>(((j >> 2) & 1) ^ 1),
                                       a.spin, abort_flag)) {
                    record_timeout(a, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * a.Nacc);
                for (int kb = 0; kb < a.d_blocks; ++kb) {
                    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, a.spin, abort_flag)) {
                        record_timeout(a, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = k_ring + stage * kKBlockBytes;
                    const uint32_t b_addr = q_buf + qb * q_stage_bytes + kb * a.q_block_bytes;
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        tc_mma_bf16(d_tmem, smem_desc_sw128(a_addr + 32 * k4),
                                    smem_desc_sw128(b_addr + 32 * k4), idesc, (kb | k4) != 0);
                    }
                    any_mma = true;
                    tc_commit(bar_empty + 8 * stage);
                    if (++stage == a.stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(bar_tfull + 8 * acc);
            }
            // drain: all MMAs issued by this thread complete before TMEM is freed
            if (any_mma) {
                tc_commit(bar_drain);
                mbar_wait_spin(bar_drain, 0, kDrainSpin);
            }
        }
    } else {
        // epilogue warpgroups; the per-segment counters they update are
        // zeroed by the prep kernel
        if (epi_wait) grid_dep_wait();
        const int e = warp >> 2;          // warpgroup: tiles j with j % 2 == e
        const int qw = warp & 3;          // TMEM lane quarter
        const int bar_id = 1 + e;
        const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
        uint8_t* out_buf = smem + L.out_buf + e * NH * kStageOutBytes;
        const uint32_t out_addr = smem_u32(out_buf);
        float2* st_sm = stats + e * 4 * 64;
        // the scratch is stored with the evict-first policy: on the larger
        // workloads it outgrows L2 and would otherwise push out every other
        // line, the kernels' code included (serving batch 250.0 -> 241.0 us
        // per call, long workload 251.0 -> 245.2; 2B unchanged)
        const uint64_t store_pol = policy_evict_first();
        volatile int* seg_flag = reinterpret_cast<volatile int*>(smem + L.seg_flag) + e;
        const int tl = qw * 32 + lane;   // token row of the tile
        // running softmax statistics of row hh * 32 + lane over this warp's
        // tokens of the current segment: (reference max, sum of exp2(y - max))
        float2 run[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) run[hh] = make_float2(-INFINITY, 0.0f);
        int64_t cur_key = -1;
        bool stores = false;
        bool ok = true;
        int64_t j = 0;
        ItemCursor cur;
        cur.tb = tb;
        cur.so = so;
        for (int64_t w = w_begin; w < w_end; ++w, ++j) {
            if (w == w_begin) cur.set(a, w, T);
            else cur.next(a, w, T);
            const Item& it = cur.it;
            const int64_t key = static_cast<int64_t>(it.slab) * a.B + it.b;
            if (key != cur_key) {
                if (cur_key >= 0) {
                    flush_rows<NH>(run, st_sm, qw, bar_id, a.rec + ((cta + cur_key) * 2 + e) * a.Rs, a.R);
                    segment_done(tb, a.B, a.nslab, C, cur_key, 1, a.rec, a.seg_cnt, a.lse2,
                                 a.R, a.Rs, st_sm, seg_flag, qw, bar_id);
                }
                cur_key = key;
            }
            if (static_cast<int>(j & 1) != e) continue;
            // all 128 threads of the warpgroup take the same decision, so the
            // named barriers below never wait for a thread that left
            const int acc = static_cast<int>(j & (kAcc - 1));
            const bool got = mbar_wait_bounded(bar_tfull + 8 * acc, static_cast<uint32_t>((j >> 2) & 1),
                                               a.spin, abort_flag);
            if (!bar_sync_and(bar_id, 128, got)) {
                record_timeout(a, abort_flag);
                ok = false;
                break;
            }
            tc_fence_after();
            float v[NH][32];
            const uint32_t taddr = tmem_base + lane_base + static_cast<uint32_t>(acc * a.Nacc);
            tmem_ld_32x32b_x32(taddr, v[0]);
            if (NH > 1) tmem_ld_32x32b_x32(taddr + 32, v[NH - 1]);
            tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < NH; ++hh)
#pragma unroll
                for (int r = 0; r < 32; ++r)  // columns past the MMA width hold no result
                    if (hh * 32 + r >= a.Nmma) v[hh][r] = 0.0f;
            const bool valid = tl < it.nvalid;
            // row maxima M of the scaled logits over the warp quarter's valid
            // tokens (rounding is monotonic, so scaling the maximum of the
            // raw dot products gives the maximum of the scaled ones)
            float m_own[NH];
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
#pragma unroll
                for (int r = 0; r < 32; ++r) v[hh][r] = valid ? v[hh][r] : -INFINITY;
                m_own[hh] = warp_rows_reduce<true>(v[hh]) * a.scale2;
                if (hh * 32 + lane < a.Rs)
                    a.lmax[((static_cast<int64_t>(it.slab) * a.tiles_max + it.tile) * 4 + qw) * a.Rs + hh * 32 +
                           lane] = m_own[hh];
            }
            // the reduction consumed the values: read the accumulator again, then free it
            tmem_ld_32x32b_x32(taddr, v[0]);
            if (NH > 1) tmem_ld_32x32b_x32(taddr + 32, v[NH - 1]);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bar_tempty + 8 * acc);

            // quantised row against M, and exp2(y - M) of the valid tokens for
            // the quarter's softmax partial
            if (qw == 0 && lane == 0 && stores) bulk_wait_read0();
            asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
            // the warp's row maxima in quantiser units, 2^11 M (lane r: row
            // hh * 32 + r), to every lane through the warp's part of the
            // statistics scratch. With y' = 2^11 y, d = 2^11 M - y' is the
            // quantised distance before rounding (>= 0 for valid tokens;
            // the scale by 2^11 is exact) and exp2(y - M) = exp2(-d 2^-11).
            float* msm = reinterpret_cast<float*>(st_sm + qw * 64);
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) msm[hh * 32 + lane] = m_own[hh] * kLogitQuant;
            __syncwarp();
            const float s2k = a.scale2 * kLogitQuant;
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                uint32_t pk[16];
                const float4* m4 = reinterpret_cast<const float4*>(msm + hh * 32);
#pragma unroll
                for (int r = 0; r < 32; r += 4) {
                    const float4 M = m4[r / 4];
                    const float Mr[4] = {M.x, M.y, M.z, M.w};
#pragma unroll
                    for (int u = 0; u < 4; u += 2) {
                        const float d0 = __fsub_rn(Mr[u], __fmul_rn(v[hh][r + u], s2k));
                        const float d1 = __fsub_rn(Mr[u + 1], __fmul_rn(v[hh][r + u + 1], s2k));
                        // invalid tokens (never read back) may give any bits
                        pk[(r + u) / 2] = __byte_perm(quant_distance(d0), quant_distance(d1), 0x5410);
                        v[hh][r + u] = valid ? exp2_ftz(__fmul_rn(d0, -kLogitQuantInv)) : 0.0f;
                        v[hh][r + u + 1] = valid ? exp2_ftz(__fmul_rn(d1, -kLogitQuantInv)) : 0.0f;
                    }
                }
                // the staging buffer has the TMA 64-byte swizzle: 16-byte chunk c
                // of row tl sits at chunk c ^ ((tl >> 1) & 3), so the eight
                // lanes of each store phase hit distinct banks
                uint4* row = reinterpret_cast<uint4*>(out_buf + hh * kStageOutBytes + tl * 64);
                const int sw = (tl >> 1) & 3;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    row[c4 ^ sw] = make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
                // lane r: this tile's (M, sum) of row hh * 32 + r, merged into the running pair
                const float z = warp_rows_reduce<false>(v[hh]);
                run[hh] = merge_partial(run[hh], make_float2(m_own[hh], z));
            }
            fence_proxy_async_smem();
            asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory");
            if (qw == 0 && lane == 0) {
                const int y = it.tile * kTileTokens;
#pragma unroll
                for (int hh = 0; hh < NH; ++hh)
                    tma_store_3d(tmap_s, out_addr + hh * kStageOutBytes, hh * 32, y, it.slab, store_pol);
                bulk_commit();
                stores = true;
            }
        }
        if (ok && cur_key >= 0) {
            flush_rows<NH>(run, st_sm, qw, bar_id, a.rec + ((cta + cur_key) * 2 + e) * a.Rs, a.R);
            segment_done(tb, a.B, a.nslab, C, cur_key, 1, a.rec, a.seg_cnt, a.lse2, a.R,
                         a.Rs, st_sm, seg_flag, qw, bar_id);
        }
        if (qw == 0 && lane == 0 && stores) bulk_wait0();
    }

}

// ------------------------------------------------------------------ host

struct LogitsMaps {
    CUtensorMap k, q, s;
};

// Tensor maps of the keys, queries and the wave's logits scratch.
cudaError_t make_logits_maps(const Plan& pl, const sp_shape* s, const uint16_t* q, const uint16_t* k,
                             void* ws, int nslab, LogitsMaps* m);

// Ring stages, dynamic shared memory and 32-row halves (1 or 2) of the
// logits phase for this plan.
cudaError_t logits_smem(const Plan& pl, int* stages, uint32_t* smem, int* nh);

// Kernel arguments and shared-memory size of the logits phase for the
// slabs [slab0, slab0 + nslab); *nh = 1 or 2 (32-row halves of the rows).
cudaError_t logits_config(const Plan& pl, const int32_t* seq_off, void* ws, int slab0, int nslab,
                          TcArgs* a, uint32_t* smem, int* nh);

}  // namespace sp

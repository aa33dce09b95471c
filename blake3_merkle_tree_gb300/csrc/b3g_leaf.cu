// b3g_leaf.cu -- leaf kernels: chunk compression fused with the CTA subtree.
//
// Source page: "BLAKE3 GPU 400x faster hashing" (qfminer.top).
//   section "Kernel 1": each CTA takes 2^t consecutive chunks, one consumer thread
//     per chunk, and reduces their CVs to one subtree CV without a round trip
//     through global memory; a producer loads the data with the tensor memory
//     accelerator (TMA).
//   section "TMA 加载": global memory is viewed as a (chunks, 256) matrix of 32-bit
//     words; one load brings a (2^t, words-per-load) tile, 128 bytes of every chunk.
//   section "消费者循环": consumers wait for a stage, read it with 128-bit shared
//     loads, compress, and release the stage to the producer.
//   section "共享内存布局与 Swizzle": stage buffers are swizzled so that the
//     consumers' row reads avoid bank conflicts.
//   section "不完整块的处理": the last CTA may hold fewer chunks, and the last chunk
//     may be partial; the partial chunk is zero padded.
//
// GB300 design (differences from the page's Hopper design):
//   - Persistent CTAs: the grid is sized to the resident capacity and each CTA walks
//     tiles blockIdx.x, blockIdx.x + gridDim.x, ...; the stage rings keep running
//     across tiles, so the copies of the next tile are in flight while the previous
//     tile's subtree is reduced.
//   - No producer threads: each consumer warp feeds itself.  Its lane 0 keeps a few
//     bulk tensor copies of the warp's own 32 chunk rows in flight in a private
//     ring and refills a stage as soon as the warp has read it, so no warp waits
//     for another warp's progress (the page uses 128 producer threads and a
//     consumer-wide barrier per stage).
//   - One reducer warp per CTA turns the consumers' chunk CVs into the tile CV,
//     taking them through two node buffers so that the consumers go on with the
//     next tile at once; the top levels of several full tiles are reduced together
//     so that those levels keep whole warps busy.
//   - The box height is at most 256 rows (the TMA limit), so one tensor map and one
//     pipeline cover every tile size up to 256 chunks; no dual pipeline is needed.
//   - The partial last chunk is not padded inside the stage: rows past the last full
//     chunk are outside the tensor map, which the TMA fills with zeros, and the one
//     thread that owns the partial chunk reads its bytes from global memory with
//     bounds checks (zero beyond the end of the input).
//   - Every barrier wait is bounded in time; a wait that gives up sets the device
//     status word and the CTA leaves after draining its copies in flight.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "b3g_device.cuh"
#include "b3g_internal.h"

// Unroll factor of the consumer's copy loop (the copies of one chunk), and the
// minimum resident CTAs per SM asked of the register allocator (0: none).
#ifndef B3G_UNROLL
#define B3G_UNROLL 1
#endif
#ifndef B3G_MIN_BLOCKS
#define B3G_MIN_BLOCKS 0
#endif
#if B3G_MIN_BLOCKS > 0
#define B3G_LEAF_BOUNDS(threads) __launch_bounds__(threads, B3G_MIN_BLOCKS)
#else
#define B3G_LEAF_BOUNDS(threads) __launch_bounds__(threads)
#endif
// Full tiles whose top tree levels the reducer warp runs together (0: every tile on
// its own), and whether the asynchronous-copy kernel's reducer runs each tree level as
// a called function (1) or inlined at each use (0).  As a call, that reducer holds one
// copy of the compression for all its levels instead of one per use: its code stays in
// the instruction caches, and the tree work that ends each launch runs sooner.  The
// bulk-tensor-copy kernel keeps the inlined levels (as a call its reducer would need 95
// registers, one CTA per SM fewer).
#ifndef B3G_TOP_BATCH
#define B3G_TOP_BATCH 8
#endif
#ifndef B3G_PAIR_NOINLINE
#define B3G_PAIR_NOINLINE 1
#endif

namespace b3g {

constexpr int kCopyLoopUnroll = B3G_UNROLL;
constexpr uint32_t kBarTree = 1;  // named barrier id of the consumer threads

// ---------------------------------------------------------------------------------
// Bulk-tensor-copy (TMA) kernel.
//   warps 0 .. C/32-1   consumers: thread r compresses chunk tile*C + r (16 chained
//                       compressions).  Each consumer warp feeds itself: its lane 0
//                       keeps S bulk tensor copies of the warp's own 32 chunk rows
//                       (LOAD bytes of each row per copy) in flight in a private ring
//                       of S stages, and refills a stage right after the warp has
//                       consumed it.  No warp waits for another warp's progress.
//   warp  C/32          reducer: reduces each tile's C chunk CVs to the tile CV.
// The consumers hand their chunk CVs to the reducer through two node buffers
// (tile k uses buffer k&1) guarded by mbarriers, so a consumer never waits for the
// tree of the previous tile: it stores its CV, arrives, and starts the next tile.
//
//   C          consumers = chunks per tile (2^t), a multiple of 32, at most 256
//   S          stages in each consumer warp's ring
//   LOAD       bytes of every chunk brought by one copy (128 or 64)
//   CHUNK_CVS  write every chunk CV instead of reducing the tile (no reducer work)
// ---------------------------------------------------------------------------------
template <int C, int S, int LOAD, bool CHUNK_CVS, uint32_t STAGE = 32 * LOAD>
struct TmaCfg {
    static_assert(C % 32 == 0 && C >= 32 && C <= 256, "consumer count");
    static_assert(LOAD == 128 || LOAD == 64, "load width");
    static constexpr int kC = C;
    static constexpr int kLoadsPerChunk = 1024 / LOAD;
    static constexpr int kBlocksPerLoad = LOAD / 64;
    static constexpr int kConsumerWarps = C / 32;
    static constexpr int kReducerWarp = kConsumerWarps;
    static constexpr int kThreads = C + 32;
    static constexpr uint32_t kRowsPerCopy = 32;                    // one warp's rows
    static constexpr uint32_t kStageBytes = STAGE;  // the bulk tensor copy's box bytes: 32 rows x LOAD
    static constexpr uint32_t kRingBytes = S * kStageBytes;
    static constexpr uint32_t kNodeBytes = C * 32;            // one node buffer
    static constexpr uint32_t kScratch1Bytes = (C / 2) * 32;  // odd tree levels
    static constexpr uint32_t kScratch2Bytes = (C / 4) * 32;  // even tree levels
    // the top five levels (32 nodes -> 1) of kTopBatch full tiles are reduced
    // together, in two ping-pong buffers of 32 and 16 nodes per tile.  Only for
    // 128-chunk tiles: smaller tiles serve small inputs (about one tile per CTA), and
    // with 256-chunk tiles the buffers would cost a resident CTA per SM.
    static constexpr uint32_t kTopBatch = (CHUNK_CVS || C != 128) ? 0 : B3G_TOP_BATCH;
    static constexpr uint32_t kTopABytes = kTopBatch * 32 * 32;
    static constexpr uint32_t kTopBBytes = kTopBatch * 16 * 32;
    // The scratch buffers (a tile's own levels) and top B (the batched levels) are
    // never in use at the same time: the reducer warp runs one or the other, so the
    // scratch lives inside top B when it fits.
    static constexpr bool kScratchInTopB = kTopBatch > 0 && kTopBBytes >= kScratch1Bytes + kScratch2Bytes;
    // layout: [align 1024][rings][2 node buffers][top A][top B][scratch 1][scratch 2][barriers]
    static constexpr uint32_t kOffNodes = kConsumerWarps * kRingBytes;
    static constexpr uint32_t kOffTopA = kOffNodes + 2 * kNodeBytes;
    static constexpr uint32_t kOffTopB = kOffTopA + kTopABytes;
    static constexpr uint32_t kOffScratch1 = kScratchInTopB ? kOffTopB : kOffTopB + kTopBBytes;
    static constexpr uint32_t kOffScratch2 = kOffScratch1 + kScratch1Bytes;
    static constexpr uint32_t kOffBars =
        kScratchInTopB ? kOffTopB + kTopBBytes : kOffScratch2 + kScratch2Bytes;
    static constexpr uint32_t kNumBars = kConsumerWarps * S + 4;
    static constexpr size_t kSmemBytes = 1024 + size_t(kOffBars) + 8 * kNumBars;
    static_assert(S >= 2 && S <= kLoadsPerChunk, "stage count");
};

struct Words8 {
    uint32_t w[8];
};

// CV of the partial last chunk (`bytes` < 1024, at least 1, starting at byte `off`),
// read straight from global memory with bounds checks.  Only the one thread that owns
// that chunk calls it, once, so it is kept out of line, away from the hot loop; all
// arguments and the result travel by value so that no caller array escapes.
// `last_flags` is the flag word of the chunk's last block: the mode bits with
// CHUNK_END (and ROOT); the blocks before it carry the mode bits alone.
__device__ __noinline__ Words8 partial_chunk_cv(const uint8_t *in, uint64_t len, uint64_t off, uint64_t ctr,
                                                uint32_t bytes, uint32_t last_flags, Words8 key) {
    const uint32_t nblocks = (bytes + 63u) / 64u;
    const uint32_t mode_flags = last_flags & ~(kChunkEnd | kRoot);
    Words8 cv = key;
    for (uint32_t b = 0; b < nblocks; ++b) {
        uint32_t m[16];
        load_block_global(in, len, off + 64ull * b, m);
        const bool last = b + 1 == nblocks;
        const uint32_t flags = (last ? last_flags : mode_flags) | (b == 0 ? kChunkStart : 0u);
        compress(cv.w, m, static_cast<uint32_t>(ctr), static_cast<uint32_t>(ctr >> 32),
                 last ? bytes - 64u * (nblocks - 1u) : 64u, flags);
    }
    return cv;
}

// One tree level in shared memory: node j of `dst` = parent(node 2j, node 2j+1 of
// `src`) for j < half, the lanes of the calling warp striding over j.
__device__ __forceinline__ void pair_level_inline(uint32_t src, uint32_t dst, uint32_t half, Words8 key,
                                                  uint32_t mode_flags) {
    const uint32_t lane = threadIdx.x & 31u;
    for (uint32_t j = lane; j < half; j += 32) {
        uint32_t l[8], r[8], p[8];
        load_node(src, 2 * j, l);
        load_node(src, 2 * j + 1, r);
        parent(key.w, mode_flags, l, r, false, p);
        store_node(dst, j, p);
    }
}

// The same level as a called function.
__device__ __noinline__ void pair_level_call(uint32_t src, uint32_t dst, uint32_t half, Words8 key,
                                             uint32_t mode_flags) {
    pair_level_inline(src, dst, half, key, mode_flags);
}

// The level as the reducer of configuration CALL runs it.
template <bool CALL>
__device__ __forceinline__ void pair_level(uint32_t src, uint32_t dst, uint32_t half, Words8 key,
                                           uint32_t mode_flags) {
    if constexpr (CALL)
        pair_level_call(src, dst, half, key, mode_flags);
    else
        pair_level_inline(src, dst, half, key, mode_flags);
}

// Fused final reduction (at most 32 tiles, one tile per CTA).  Called by a whole
// reducer warp right after its lane 0 stored the tile CV.  The warp that draws the
// last ticket has seen every other tile CV published (each is stored, then fenced,
// before its warp takes a ticket) and folds them with the warp-level tree, ROOT on
// the final compression.  This replaces the separate reduction launch for small inputs.
__device__ __forceinline__ void fused_final_reduce(const LeafArgs &a, const uint32_t key[8], uint32_t mode_flags) {
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t ticket = 0;
    if (lane == 0) {
        __threadfence();
        ticket = atomicAdd(a.ticket, 1u);
    }
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    const uint32_t n = static_cast<uint32_t>(a.n_tiles);
    if (ticket != n - 1) return;
    __threadfence();
    uint32_t x[8];
    if (lane < n) {
        const uint4 *p = reinterpret_cast<const uint4 *>(a.out + 32ull * lane);
        const uint4 w0 = __ldcg(p), w1 = __ldcg(p + 1);
        x[0] = w0.x; x[1] = w0.y; x[2] = w0.z; x[3] = w0.w;
        x[4] = w1.x; x[5] = w1.y; x[6] = w1.z; x[7] = w1.w;
    }
    warp_tree(x, n, key, mode_flags, a.root != 0);
    if (lane == 0) {
        uint4 *o = reinterpret_cast<uint4 *>(a.final_out);
        o[0] = make_uint4(x[0], x[1], x[2], x[3]);
        o[1] = make_uint4(x[4], x[5], x[6], x[7]);
    }
}

// Tile index ring of the asynchronous-copy kernel: at the start of its k-th tile
// (counting from 0) the CTA publishes its (k + 1)-th tile in slot k mod kTileSlots, and
// barrier k mod kTileSlots completes once per publication (parity (k / kTileSlots) & 1).
// Four slots suffice: slot k mod 4 is rewritten at the start of tile k + 4, which the
// publishing warp reaches only after the node buffer of tile k + 2 was handed over, so
// after every consumer warp (which reads the slot during tile k) and the reducer (after
// tile k) have read it.
constexpr uint32_t kTileSlots = 4;

// The reducer warp of the leaf kernels (page sections "Merkle Tree 归约" and "未来工作"):
// turns each tile's chunk CVs, handed over in node buffer k & 1, into the tile CV.  The
// CTA's tiles are blockIdx.x, blockIdx.x + gridDim.x, ... (`slots` == 0) or the ones
// published in the tile index ring at `slots` (the first is blockIdx.x): the tile after
// the k-th was published before the consumers' hand-over of the k-th, which the reducer
// has waited for, so reading it needs no further wait.
template <typename Cfg, uint32_t MODE, bool PAIR_CALL = false>
__device__ __forceinline__ void reducer_warp(const LeafArgs &a, const uint32_t key[8], uint32_t rings0,
                                             uint32_t nodes0, uint32_t cvfull0, uint32_t cvempty0,
                                             uint32_t slots = 0) {
    constexpr int C = Cfg::kC;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t scratch1 = rings0 + Cfg::kOffScratch1;
    const uint32_t scratch2 = rings0 + Cfg::kOffScratch2;

    const uint32_t topA = rings0 + Cfg::kOffTopA;
    const uint32_t topB = rings0 + Cfg::kOffTopB;
    Words8 key8;
#pragma unroll
    for (int i = 0; i < 8; ++i) key8.w[i] = key[i];
    // Full tiles are reduced down to 32 nodes each, which wait side by side in
    // top A; every kTopBatch tiles the top levels of all of them run as one
    // array (pairing never mixes two tiles: each holds a power-of-two count),
    // so those levels keep whole warps busy instead of 16, 8, 4, 2 and 1 lanes.
    uint32_t pending = 0;  // tiles waiting in top A
    uint64_t my_tile = 0;  // lane p: the index of pending tile p
    auto flush = [&]() {
        if (pending == 0) return;
        uint32_t n = pending * 32u, src = topA, dst = topB;
        while (n > pending) {
            pair_level<PAIR_CALL>(src, dst, n >> 1, key8, MODE);
            __syncwarp();
            const uint32_t t = src;
            src = dst;
            dst = t;
            n >>= 1;
        }
        if (lane < pending) {
            uint32_t x[8];
            load_node(src, lane, x);
            uint4 *o = reinterpret_cast<uint4 *>(a.out + my_tile * 32);
            o[0] = make_uint4(x[0], x[1], x[2], x[3]);
            o[1] = make_uint4(x[4], x[5], x[6], x[7]);
        }
        __syncwarp();
        pending = 0;
    };
    uint32_t k = 0;
    for (uint64_t tile = blockIdx.x; tile < a.n_tiles; ++k) {
        const uint32_t b = k & 1u;
        const uint32_t src0 = nodes0 + b * Cfg::kNodeBytes;
        if (!mbar_wait_bounded(cvfull0 + 8 * b, (k >> 1) & 1u, a.wait_limit_ns)) {
            atomicOr(a.status, B3G_DEVICE_STATUS_TIMEOUT);
            break;
        }
        const uint64_t rem = a.n_chunks - tile * C;
        uint32_t cnt = rem < C ? static_cast<uint32_t>(rem) : static_cast<uint32_t>(C);
        if (Cfg::kTopBatch > 0 && cnt == C && !a.ticket && !(a.root && a.n_tiles == 1)) {
            // a full tile: its levels down to 32 nodes, the last into top A
            const uint32_t slot = topA + pending * 1024u;
            uint32_t src = src0, level = 0;
            for (uint32_t n = C; n > 32; n >>= 1, ++level) {
                const uint32_t dst = n == 64 ? slot : ((level & 1u) ? scratch2 : scratch1);
                pair_level<PAIR_CALL>(src, dst, n >> 1, key8, MODE);
                __syncwarp();
                if (level == 0) mbar_arrive(cvempty0 + 8 * b);  // node buffer read
                src = dst;
            }
            if (level == 0) {  // 32 chunks per tile: the node buffer is the top level
                uint32_t x[8];
                load_node(src0, lane, x);
                __syncwarp();
                mbar_arrive(cvempty0 + 8 * b);
                store_node(slot, lane, x);
                __syncwarp();
            }
            if (lane == pending) my_tile = tile;
            if (++pending == Cfg::kTopBatch) flush();
            tile = slots ? lds64(slots + 8 * (k % kTileSlots)) : tile + gridDim.x;
            continue;
        }
        // a partial tile, a single-tile root or the fused final reduction: on its own
        flush();
        uint32_t src = src0;
        uint32_t level = 0;
        // Levels with more than 32 nodes: pairs (2j, 2j+1) -> node j,
        // ping-ponging between two scratch buffers; an odd last node moves up
        // unchanged.
        while (cnt > 32) {
            const uint32_t dst = (level & 1u) ? scratch2 : scratch1;
            const uint32_t half = cnt >> 1;
            pair_level<PAIR_CALL>(src, dst, half, key8, MODE);
            if ((cnt & 1u) && lane == 0) {
                uint32_t t[8];
                load_node(src, cnt - 1, t);
                store_node(dst, half, t);
            }
            __syncwarp();
            if (level == 0) mbar_arrive(cvempty0 + 8 * b);  // node buffer read
            src = dst;
            cnt = (cnt + 1) >> 1;
            ++level;
        }
        uint32_t x[8];
        if (lane < cnt) load_node(src, lane, x);
        __syncwarp();
        if (level == 0) mbar_arrive(cvempty0 + 8 * b);
        warp_tree(x, cnt, key, MODE, a.root && a.n_tiles == 1);
        if (lane == 0) {
            uint4 *o = reinterpret_cast<uint4 *>(a.out + tile * 32);
            o[0] = make_uint4(x[0], x[1], x[2], x[3]);
            o[1] = make_uint4(x[4], x[5], x[6], x[7]);
        }
        if (a.ticket) fused_final_reduce(a, key, MODE);
        tile = slots ? lds64(slots + 8 * (k % kTileSlots)) : tile + gridDim.x;
    }
    flush();
}

// The reducer warp as a called function, for the asynchronous-copy kernel: inlined
// there, the tree code's registers and the consumers' fetch state compete in one
// allocation and ptxas spills (52 bytes of reloads at five CTAs per SM); called, the
// kernel keeps 72 registers and the aligned kernel spills nothing.
template <typename Cfg, uint32_t MODE>
__device__ __noinline__ void reducer_warp_call(const LeafArgs &a, const uint32_t *key, uint32_t rings0,
                                               uint32_t nodes0, uint32_t cvfull0, uint32_t cvempty0,
                                               uint32_t slots) {
    uint32_t k8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) k8[i] = key[i];
    reducer_warp<Cfg, MODE, B3G_PAIR_NOINLINE != 0>(a, k8, rings0, nodes0, cvfull0, cvempty0, slots);
}

// End of a consumer thread's tile: the owner of the partial last chunk redoes it from
// global memory (its row in the stage was not that chunk's bytes), then the chunk CV is
// written out (CHUNK_CVS) or handed to the reducer: wait until node buffer k & 1 is free
// (the reducer has read tile k - 2), store, arrive.  Returns false if that wait gave up.
template <typename Cfg, bool CHUNK_CVS, uint32_t MODE>
__device__ __forceinline__ bool finish_tile(const LeafArgs &a, const uint32_t key[8], uint32_t cv[8],
                                            uint64_t chunk, uint64_t ctr, uint32_t end_flags, uint32_t k,
                                            uint32_t nodes0, uint32_t cvfull0, uint32_t cvempty0) {
    const bool valid = chunk < a.n_chunks;
    if (a.tail_bytes != 0 && chunk == a.n_full) {
        Words8 k8, t;
#pragma unroll
        for (int i = 0; i < 8; ++i) k8.w[i] = key[i];
        t = partial_chunk_cv(a.in, a.len, chunk * kChunkBytes, ctr, a.tail_bytes, MODE | end_flags, k8);
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[i] = t.w[i];
    }
    if constexpr (CHUNK_CVS) {
        if (valid) {
            uint4 *o = reinterpret_cast<uint4 *>(a.out + chunk * 32);
            o[0] = make_uint4(cv[0], cv[1], cv[2], cv[3]);
            o[1] = make_uint4(cv[4], cv[5], cv[6], cv[7]);
        }
    } else {
        const uint32_t b = k & 1u;
        if (k >= 2 && !mbar_wait_bounded(cvempty0 + 8 * b, ((k >> 1) - 1) & 1u, a.wait_limit_ns)) {
            atomicOr(a.status, B3G_DEVICE_STATUS_TIMEOUT);
            return false;
        }
        if (valid) store_node(nodes0 + b * Cfg::kNodeBytes, threadIdx.x, cv);
        mbar_arrive(cvfull0 + 8 * b);
    }
    return true;
}

template <int C, int S, int LOAD, bool CHUNK_CVS, uint32_t MODE>
__global__ void B3G_LEAF_BOUNDS(C + 32)
    leaf_tma_kernel(const __grid_constant__ CUtensorMap tmap, const LeafArgs a) {
    using Cfg = TmaCfg<C, S, LOAD, CHUNK_CVS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t rings0 = (raw + 1023u) & ~1023u;
    const uint32_t nodes0 = rings0 + Cfg::kOffNodes;  // buffer b at nodes0 + b * kNodeBytes
    const uint32_t full0 = rings0 + Cfg::kOffBars;               // S barriers per consumer warp
    const uint32_t cvfull0 = full0 + 8 * Cfg::kConsumerWarps * S;  // 2: node buffer b is filled
    const uint32_t cvempty0 = cvfull0 + 16;                        // 2: node buffer b is free

    const uint32_t tid = threadIdx.x;
    const uint32_t warp = tid >> 5;
    const uint32_t lane = tid & 31u;

    // launched early behind the previous kernel of the stream: no global-memory access
    // before it has finished (it may still read this launch's output buffer)
    grid_dependency_wait();
    if (tid == 0) {
        // the reduction launched behind this kernel may start now: its CTAs take the
        // places of finished CTAs and wait for this grid's results
        launch_dependents();
        for (int i = 0; i < Cfg::kConsumerWarps * S; ++i) mbar_init(full0 + 8 * i, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(cvfull0 + 8 * b, C);
            mbar_init(cvempty0 + 8 * b, 32);
        }
        fence_mbar_init();
    }
    __syncthreads();

    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = a.key[i];

    if (warp == Cfg::kReducerWarp) {
        // -------------------------------- reducer --------------------------------
        if constexpr (!CHUNK_CVS) reducer_warp<Cfg, MODE>(a, key, rings0, nodes0, cvfull0, cvempty0);
        return;
    }

    // --------------------------------- consumers ---------------------------------
    const uint32_t r = tid;
    const uint32_t ring = rings0 + warp * Cfg::kRingBytes;
    const uint32_t fullw = full0 + 8 * S * warp;
    // 16-byte unit u of row `lane` sits at u ^ swz (TMA 128B / 64B swizzle); the byte
    // offsets of the row's units within a stage are fixed for the thread
    const uint32_t swz = LOAD == 128 ? (lane & 7u) : ((lane >> 1) & 3u);
    uint32_t unit_addr[LOAD / 16];
#pragma unroll
    for (int u = 0; u < LOAD / 16; ++u) unit_addr[u] = ring + lane * LOAD + ((static_cast<uint32_t>(u) ^ swz) << 4);

    // Copy stream of this warp: copy i brings part (i mod kLoadsPerChunk) of the warp's
    // 32 rows of the CTA's (i / kLoadsPerChunk)-th tile.  Only lane 0 issues.
    const uint64_t my_tiles = a.n_tiles > blockIdx.x ? (a.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    uint32_t copies_left = static_cast<uint32_t>(my_tiles * Cfg::kLoadsPerChunk);
    uint32_t next_row = static_cast<uint32_t>(blockIdx.x * C + Cfg::kRowsPerCopy * warp);
    const uint32_t row_step = gridDim.x * C;
    uint32_t next_part = 0;
    uint32_t issued = 0, consumed = 0;
    auto issue = [&](uint32_t stage) {
        if (copies_left == 0) return;
        --copies_left;
        mbar_arrive_expect_tx(fullw + 8 * stage, Cfg::kStageBytes);
        tma_load_2d(ring + stage * Cfg::kStageBytes, &tmap, static_cast<int32_t>(next_part * (LOAD / 4)),
                    static_cast<int32_t>(next_row), fullw + 8 * stage);
        ++issued;
        if (++next_part == Cfg::kLoadsPerChunk) {
            next_part = 0;
            next_row += row_step;
        }
    };
    if (lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap) : "memory");
        for (int i = 0; i < S; ++i) issue(static_cast<uint32_t>(i));
    }

    // When S divides the copies per chunk every chunk starts at stage 0, so a copy's
    // stage and fill parity follow from its position in the chunk (and the loop may be
    // unrolled so that stage addresses become immediates).
    constexpr bool kStageFromPos = Cfg::kLoadsPerChunk % S == 0;
    uint32_t s = 0, ph = 0;  // otherwise: stage of the next copy and its fill parity
    uint32_t k = 0;
    bool aborted = false;

    for (uint64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++k) {
        const uint64_t chunk = tile * C + r;
        const bool valid = chunk < a.n_chunks;
        const uint64_t ctr = a.counter_base + chunk;
        const uint32_t ctr_lo = static_cast<uint32_t>(ctr);
        const uint32_t ctr_hi = static_cast<uint32_t>(ctr >> 32);
        const uint32_t end_flags = kChunkEnd | ((a.root && a.n_chunks == 1) ? kRoot : 0u);
        const uint32_t tile_par = (k * (Cfg::kLoadsPerChunk / S)) & 1u;  // used when kStageFromPos

        // Every thread compresses its row as a full chunk; the owner of the partial
        // last chunk (its row reads as zeros) redoes its chunk after the loop.
        uint32_t cv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[i] = key[i];
        uint32_t flags = MODE | kChunkStart;

#pragma unroll kCopyLoopUnroll
        for (int ld = 0; ld < Cfg::kLoadsPerChunk; ++ld) {
            const uint32_t st = kStageFromPos ? static_cast<uint32_t>(ld % S) : s;
            const uint32_t par = kStageFromPos ? (tile_par ^ (static_cast<uint32_t>(ld / S) & 1u)) : ph;
            if (!mbar_wait_bounded(fullw + 8 * st, par, a.wait_limit_ns)) {
                atomicOr(a.status, B3G_DEVICE_STATUS_TIMEOUT);
                aborted = true;
                break;
            }
            const uint32_t stage_off = st * Cfg::kStageBytes;
#pragma unroll
            for (int j = 0; j < Cfg::kBlocksPerLoad; ++j) {
                const int b = ld * Cfg::kBlocksPerLoad + j;
                uint32_t m[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = lds128(unit_addr[4 * j + q] + stage_off);
                    m[4 * q + 0] = w.x;
                    m[4 * q + 1] = w.y;
                    m[4 * q + 2] = w.z;
                    m[4 * q + 3] = w.w;
                }
                compress(cv, m, ctr_lo, ctr_hi, 64u, b == 15 ? (flags | end_flags) : flags);
                flags = MODE;
            }
            // every lane has consumed stage st (its words went into the compression):
            // refill it with the copy S positions ahead
            __syncwarp();
            ++consumed;
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(st);
            }
            if (!kStageFromPos && ++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (aborted) break;
        if (!finish_tile<Cfg, CHUNK_CVS, MODE>(a, key, cv, chunk, ctr, end_flags, k, nodes0, cvfull0, cvempty0)) {
            aborted = true;
            break;
        }
    }
    // After a give-up, wait (bounded) for this warp's copies still in flight, so that
    // none lands in shared memory after the CTA has left.  Without a give-up every
    // copy issued has been consumed.
    if (aborted && lane == 0) {
        for (uint32_t i = consumed; i < issued; ++i) {
            const uint32_t st = i % S;
            mbar_wait_bounded(fullw + 8 * st, (i / S) & 1u, a.wait_limit_ns);
        }
    }
}

// ---------------------------------------------------------------------------------
// Asynchronous-copy kernel: the same tiles, reducer warp and node buffers as the
// bulk-tensor-copy kernel; only the staging differs.  Every lane of a consumer warp
// copies 16-byte units of the warp's own 32 chunk rows with cp.async: copy i of lane l
// brings unit l >> 3 (of the four of a 64-byte block) of row (l & 7) + 8 i, so that
// one copy instruction reads 8 rows x 64 contiguous bytes.  A stage is laid out
// unit-major, [unit 0..3][row 0..31][16 bytes]: an instruction's copies land in four
// runs of 128 contiguous bytes, and lane r's four 128-bit reads of its row are 512
// bytes apart, so neither side has bank conflicts and no swizzle is needed.  Each lane
// waits for its own copy groups (cp.async.wait_group, a hardware wait for the thread's
// own copies) and a warp barrier makes the other lanes' copies visible; all lanes
// refill a stage right after the warp has read it.  No elected lane, no mbarrier and
// no tensor map on the data path.
//   S  stages in each consumer warp's ring, 2 KiB each (one 64-byte block of 32 rows)
// ---------------------------------------------------------------------------------
template <int C, int S, bool MIS>
struct AsyncCfg {
    // a stage holds 4 16-byte units of each of the 32 rows, 5 for a misaligned input
    static constexpr uint32_t kUnits = MIS ? 5 : 4;
    using Base = TmaCfg<C, S, 64, false, kUnits * 512>;
    // rings, node buffers and reducer buffers as in the bulk-tensor-copy kernel, then
    // the 4 node-buffer barriers, the 4 tile-slot barriers and the 4 tile slots,
    // aligned to 128 bytes
    static constexpr size_t kSmemBytes = 128 + size_t(Base::kOffBars) + 96;
};

// Resident CTAs per SM asked of the register allocator for the asynchronous-copy
// kernel: 5 for 128-chunk tiles (at most 80 registers; the consumers need 56, the
// reducer's tree code drives the count), none otherwise.
#ifndef B3G_ASYNC_MIN_BLOCKS
#define B3G_ASYNC_MIN_BLOCKS 5
#endif

// Words m[0..15] of a block that starts `sh` / 8 + 4 Q bytes into the 20 words x: each
// funnel-shifted out of two neighbours (sh = 0 takes the word as it is).
template <int Q>
__device__ __forceinline__ void shifted_words(const uint32_t x[20], uint32_t sh, uint32_t m[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = __funnelshift_r(x[i + Q], x[i + Q + 1], sh);
}

// Block of a tile at which thread 0 takes the CTA's next tile from the counter (-1: at
// block 16 - S, the first one whose refill is the next tile's).
#ifndef B3G_GRAB_BLOCK
#define B3G_GRAB_BLOCK -1
#endif

template <int C, int S, bool CHUNK_CVS, uint32_t MODE, bool MIS>
__global__ void __launch_bounds__(C + 32, C == 128 ? B3G_ASYNC_MIN_BLOCKS : 1) leaf_async_kernel(const LeafArgs a) {
    constexpr uint32_t kGrabBlock = B3G_GRAB_BLOCK < 0 ? 16 - S : B3G_GRAB_BLOCK;
    static_assert(kGrabBlock <= 16 - S, "the next tile is needed at block 16 - S");
    using Cfg = TmaCfg<C, S, 64, CHUNK_CVS, AsyncCfg<C, S, MIS>::kUnits * 512>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t rings0 = (smem_u32(smem_raw) + 127u) & ~127u;
    const uint32_t nodes0 = rings0 + Cfg::kOffNodes;  // buffer b at nodes0 + b * kNodeBytes
    const uint32_t cvfull0 = rings0 + Cfg::kOffBars;  // 2: node buffer b is filled
    const uint32_t cvempty0 = cvfull0 + 16;           // 2: node buffer b is free
    const uint32_t slotbar0 = cvfull0 + 32;           // kTileSlots: tile slot s is written
    const uint32_t slots = cvfull0 + 64;              // kTileSlots tile indices

    const uint32_t tid = threadIdx.x;
    const uint32_t warp = tid >> 5;
    const uint32_t lane = tid & 31u;

    grid_dependency_wait();  // see leaf_tma_kernel
    if (tid == 0) {
        launch_dependents();
        for (int b = 0; b < 2; ++b) {
            mbar_init(cvfull0 + 8 * b, C);
            mbar_init(cvempty0 + 8 * b, 32);
        }
        for (uint32_t i = 0; i < kTileSlots; ++i) mbar_init(slotbar0 + 8 * i, 1);
        fence_mbar_init();
    }
    __syncthreads();

    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = a.key[i];

    if (warp == Cfg::kReducerWarp) {
        if constexpr (!CHUNK_CVS) reducer_warp_call<Cfg, MODE>(a, key, rings0, nodes0, cvfull0, cvempty0, slots);
        return;
    }

    // --------------------------------- consumers ---------------------------------
    const uint32_t ring = rings0 + warp * Cfg::kRingBytes;
    const uint32_t rd = ring + lane * 16u;                             // unit u of row `lane`: + 512 u
    const uint32_t wr = ring + (lane >> 3) * 512u + (lane & 7u) * 16u;  // copy i: + 128 i
    const uint32_t lrow = warp * 32u + (lane & 7u);                     // copy i: row lrow + 8 i of a tile
    // A misaligned input (MIS) is read as the 16-byte units of the aligned-down range:
    // its block b of row r lies in units 4 b .. 4 b + 4 counted from `base` + 1024 r,
    // starting `skew` bytes into the first.  Units 0..3 are copied as for an aligned
    // input; the fifth by a fifth copy per lane, of the lane's own row.  Every unit copied
    // holds at least one byte of the input, so none crosses a page the input does not
    // touch.
    const uint32_t skew = MIS ? static_cast<uint32_t>(reinterpret_cast<uintptr_t>(a.in) & 15u) : 0u;
    const uint8_t *base = a.in - skew;

    // The CTA's tiles: the first is blockIdx.x; at the start of each tile thread 0
    // takes the next one, from the zeroed counter a.tile_counter (gridDim.x + its old
    // value) or, without one, gridDim.x further on, and publishes it in the tile slot
    // ring.  A tile index of n_tiles or more ends the sequence.  With the counter the
    // tiles go to the CTAs that finish first, so every SM ends within about one tile of
    // the others whatever the placement of the CTAs on the SMs.  Every tile processed
    // takes once (the CTA's last take finds no tile), so a launch that completes takes
    // exactly n_tiles times and the last take leaves the counter at zero again.
    //
    // Fetch stream of this warp: the S blocks ahead of the one being compressed; from
    // block 16 - S of a tile on, they are the next tile's first blocks.  `fp` is the
    // lane's source of the next fetch (its unit of row lrow of that tile, at that
    // block); `full_f` says whether all 32 rows of the warp in that tile are full
    // chunks.  If not (only the input's last tile, or a tile past the end) only the
    // full-chunk rows are copied: the other rows' CVs are discarded, or recomputed from
    // global memory for the partial chunk.  Every fetch closes one copy group.
    auto warp_rows_full = [&](uint64_t t) { return t * C + warp * 32u + 32u <= a.n_full; };
    auto lane_src = [&](uint64_t t) { return base + (t * C + lrow) * kChunkBytes + (lane >> 3) * 16u; };
    // the fifth unit of the lane's own row (MIS): row warp * 32 + lane, unit 4
    const uint32_t fifth_off = (warp * 32u + lane) * static_cast<uint32_t>(kChunkBytes) + 64u -
                               (lrow * static_cast<uint32_t>(kChunkBytes) + (lane >> 3) * 16u);
    const uint32_t d5 = ring + 4u * 512u + lane * 16u;
    uint64_t tile = blockIdx.x;
    const uint8_t *fp = lane_src(tile);
    bool full_f = warp_rows_full(tile);
    auto fetch = [&](uint32_t st) {
        const uint32_t d = wr + st * Cfg::kStageBytes;
        if (full_f) {
#pragma unroll
            for (int i = 0; i < 4; ++i) cp_async16(d + 128u * i, fp + 8192u * i);
            if constexpr (MIS) cp_async16(d5 + st * Cfg::kStageBytes, fp + fifth_off);
        } else {
            const uint64_t row = static_cast<uint64_t>(fp - base) / kChunkBytes;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (row + 8u * i < a.n_full) cp_async16(d + 128u * i, fp + 8192u * i);
            if constexpr (MIS) {
                if (row - (lane & 7u) + lane < a.n_full) cp_async16(d5 + st * Cfg::kStageBytes, fp + fifth_off);
            }
        }
        cp_async_commit();
        fp += 64u;
    };
#pragma unroll
    for (int j = 0; j < S; ++j) fetch(static_cast<uint32_t>(j));

    uint32_t st = 0;  // stage of the next block
    bool aborted = false;
    for (uint32_t k = 0; tile < a.n_tiles && !aborted; ++k) {
        const uint32_t slot = k % kTileSlots;
        const uint64_t chunk = tile * C + tid;
        const uint64_t ctr = a.counter_base + chunk;
        const uint32_t ctr_lo = static_cast<uint32_t>(ctr);
        const uint32_t ctr_hi = static_cast<uint32_t>(ctr >> 32);
        const uint32_t end_flags = kChunkEnd | ((a.root && a.n_chunks == 1) ? kRoot : 0u);

        // Every thread compresses its row as a full chunk; the owner of the partial
        // last chunk redoes its chunk in finish_tile.
        uint32_t cv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[i] = key[i];
        uint32_t flags = MODE | kChunkStart;

#pragma unroll 1
        for (uint32_t b = 0; b < 16; ++b) {
            if (b == kGrabBlock && tid == 0) {
                // the next tile, taken kGrabBlock blocks into this one: late enough that
                // the CTAs that run faster take more tiles, early enough that the other
                // warps find it published when they need it (block 16 - S)
                uint64_t nt = tile + gridDim.x;
                if (a.tile_counter) {
                    // one take per tile processed, n_tiles in all: the take that returns
                    // n_tiles - 1 is the last, and puts the counter back to zero
                    const uint32_t old = atomicAdd(a.tile_counter, 1u);
                    if (old == static_cast<uint32_t>(a.n_tiles - 1)) atomicExch(a.tile_counter, 0u);
                    nt = gridDim.x + static_cast<uint64_t>(old);
                }
                sts64(slots + 8 * slot, nt);
                mbar_arrive(slotbar0 + 8 * slot);
            }
            cp_async_wait<S - 1>();  // this lane's copies of block b have landed
            __syncwarp();            // ... and every other lane's
            const uint32_t rs = rd + st * Cfg::kStageBytes;
            uint32_t m[16];
            if constexpr (MIS) {
                uint32_t x[20];
#pragma unroll
                for (int q = 0; q < 5; ++q) {
                    const uint4 w = lds128(rs + 512u * q);
                    x[4 * q + 0] = w.x;
                    x[4 * q + 1] = w.y;
                    x[4 * q + 2] = w.z;
                    x[4 * q + 3] = w.w;
                }
                const uint32_t sh = (skew & 3u) * 8u;
                switch (skew >> 2) {  // the same for every lane and block
                    case 0: shifted_words<0>(x, sh, m); break;
                    case 1: shifted_words<1>(x, sh, m); break;
                    case 2: shifted_words<2>(x, sh, m); break;
                    default: shifted_words<3>(x, sh, m); break;
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = lds128(rs + 512u * q);
                    m[4 * q + 0] = w.x;
                    m[4 * q + 1] = w.y;
                    m[4 * q + 2] = w.z;
                    m[4 * q + 3] = w.w;
                }
            }
            compress(cv, m, ctr_lo, ctr_hi, 64u, b == 15 ? (flags | end_flags) : flags);
            flags = MODE;
            __syncwarp();  // every lane has read stage st: refill it, S blocks ahead
            if (b == 16 - S) {
                // from here on the fetches are the next tile's: wait for its index
                const bool ok = mbar_wait_bounded(slotbar0 + 8 * slot, (k / kTileSlots) & 1u, a.wait_limit_ns);
                if (__any_sync(0xffffffffu, !ok)) {
                    if (lane == 0) atomicOr(a.status, B3G_DEVICE_STATUS_TIMEOUT);
                    aborted = true;
                    break;
                }
                const uint64_t next = lds64(slots + 8 * slot);
                fp = lane_src(next);
                full_f = warp_rows_full(next);
            }
            fetch(st);
            if (++st == S) st = 0;
        }
        if (aborted) break;
        // the decision to leave is the warp's, so that no lane misses a warp barrier
        const bool ok = finish_tile<Cfg, CHUNK_CVS, MODE>(a, key, cv, chunk, ctr, end_flags, k, nodes0, cvfull0,
                                                          cvempty0);
        if (__any_sync(0xffffffffu, !ok)) break;
        tile = lds64(slots + 8 * slot);  // read (after its barrier) during the last blocks
    }
    cp_async_wait<0>();  // no copy may land after the CTA has left
}

// ---------------------------------------------------------------------------------
// Plain-load kernel: any alignment, any length (including 0 and inputs without a
// full chunk).  Same tiles and subtree as the TMA kernel; each thread reads its
// chunk's blocks from global memory with bounds checks.
// ---------------------------------------------------------------------------------
template <int C, bool CHUNK_CVS, uint32_t MODE>
__global__ void __launch_bounds__(C) leaf_direct_kernel(const LeafArgs a) {
    __shared__ __align__(128) uint8_t node_mem[C * 32];
    const uint32_t nodes = smem_u32(node_mem);
    grid_dependency_wait();  // see leaf_tma_kernel
    if (threadIdx.x == 0) launch_dependents();
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = a.key[i];
    const uint32_t r = threadIdx.x;

    for (uint64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
        const uint64_t chunk = tile * C + r;
        const bool valid = chunk < a.n_chunks;
        const uint64_t start = chunk * kChunkBytes;
        const uint64_t rest = (valid && start < a.len) ? a.len - start : 0;
        const uint32_t bytes = rest < kChunkBytes ? static_cast<uint32_t>(rest) : 1024u;
        const uint32_t nblocks = bytes == 0 ? 1u : (bytes + 63u) / 64u;
        const uint32_t last_len = bytes - 64u * (nblocks - 1u);
        const uint64_t ctr = a.counter_base + chunk;
        const uint32_t end_flags = kChunkEnd | ((a.root && a.n_chunks == 1) ? kRoot : 0u);
        uint32_t cv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[i] = key[i];
        if (valid) {
            // the next block's loads are issued before this block's compression, so
            // their latency hides behind it
            uint32_t m[16];
            load_block_units(a.in, a.len, start, m);
#pragma unroll 1
            for (uint32_t b = 0; b < nblocks; ++b) {
                const bool last = b + 1 == nblocks;
                uint32_t nx[16];
                if (!last) load_block_units(a.in, a.len, start + 64ull * (b + 1), nx);
                const uint32_t flags = MODE | (b == 0 ? kChunkStart : 0u) | (last ? end_flags : 0u);
                compress(cv, m, static_cast<uint32_t>(ctr), static_cast<uint32_t>(ctr >> 32),
                         last ? last_len : 64u, flags);
                if (!last) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) m[i] = nx[i];
                }
            }
        }
        if constexpr (CHUNK_CVS) {
            if (valid) {
                uint4 *o = reinterpret_cast<uint4 *>(a.out + chunk * 32);
                o[0] = make_uint4(cv[0], cv[1], cv[2], cv[3]);
                o[1] = make_uint4(cv[4], cv[5], cv[6], cv[7]);
            }
        } else {
            if (valid) store_node(nodes, r, cv);
            named_bar_sync(kBarTree, C);
            const uint64_t rem = a.n_chunks - tile * C;
            const uint32_t cnt = rem < C ? static_cast<uint32_t>(rem) : static_cast<uint32_t>(C);
            uint32_t root_cv[8];
            block_tree(nodes, cnt, r, C, kBarTree, key, MODE, a.root && a.n_tiles == 1, root_cv);
            if (r == 0) {
                uint4 *o = reinterpret_cast<uint4 *>(a.out + tile * 32);
                o[0] = make_uint4(root_cv[0], root_cv[1], root_cv[2], root_cv[3]);
                o[1] = make_uint4(root_cv[4], root_cv[5], root_cv[6], root_cv[7]);
            }
        }
    }
}

// ---------------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------------
namespace {

constexpr int kMaxDevices = 64;

// Stage count and load width per tile size (chosen by measurement on GB300; the
// B3G_TUNE_* macros exist so that other settings can be built for comparison).
#ifndef B3G_TUNE_S256
#define B3G_TUNE_S256 3
#endif
#ifndef B3G_TUNE_LOAD256
#define B3G_TUNE_LOAD256 64
#endif
#ifndef B3G_TUNE_S128
#define B3G_TUNE_S128 2
#endif
#ifndef B3G_TUNE_LOAD128
#define B3G_TUNE_LOAD128 64
#endif
template <int C>
struct Tuning;
template <>
struct Tuning<256> {
    static constexpr int S = B3G_TUNE_S256, LOAD = B3G_TUNE_LOAD256;
};
template <>
struct Tuning<128> {
    static constexpr int S = B3G_TUNE_S128, LOAD = B3G_TUNE_LOAD128;
};
#ifndef B3G_TUNE_S64
#define B3G_TUNE_S64 4
#endif
#ifndef B3G_TUNE_LOAD64
#define B3G_TUNE_LOAD64 64
#endif
template <>
struct Tuning<64> {
    static constexpr int S = B3G_TUNE_S64, LOAD = B3G_TUNE_LOAD64;
};
template <>
struct Tuning<32> {
    static constexpr int S = 4, LOAD = 128;
};

// Staging of the leaf kernel for 16-byte aligned inputs: 1 = per-lane asynchronous
// copies (leaf_async_kernel), 0 = bulk tensor copies (leaf_tma_kernel); and the stage
// count of the asynchronous-copy rings per tile size.
#ifndef B3G_STAGING
#define B3G_STAGING 1
#endif
#ifndef B3G_ASYNC_S
#define B3G_ASYNC_S 2
#endif
template <int C>
struct AsyncTuning {
    static constexpr int S = B3G_ASYNC_S;
};

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct DeviceInfo {
    int sm_count = 0;
};

b3g_status device_info(int dev, DeviceInfo &out) {
    static std::mutex mu;
    static DeviceInfo cache[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return B3G_ERR_ARG;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sm_count == 0) {
        int sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        cache[dev].sm_count = sms;
    }
    out = cache[dev];
    return B3G_OK;
}

// Per-device, per-kernel launch set-up: the shared-memory opt-in and the number of
// resident CTAs per SM (the persistent grid is that times the SM count).
b3g_status kernel_blocks_per_sm(const void *kernel, int threads, size_t smem, int dev, int &blocks) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({kernel, dev});
    if (it != cache.end()) {
        blocks = it->second;
        return B3G_OK;
    }
    cudaError_t e;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (n < 1) return cuda_fail(cudaErrorInvalidConfiguration, "occupancy is zero");
    cache[{kernel, dev}] = n;
    blocks = n;
    return B3G_OK;
}

uint64_t grid_for(uint64_t n_tiles, int blocks_per_sm, int sms) {
    const uint64_t cap = static_cast<uint64_t>(blocks_per_sm) * static_cast<uint64_t>(sms);
    return n_tiles < cap ? n_tiles : cap;
}

template <int C, bool CV, uint32_t MODE>
b3g_status launch_tma(const LeafArgs &a, cudaStream_t stream, int dev, const DeviceInfo &info) {
    using T = Tuning<C>;
    using Cfg = TmaCfg<C, T::S, T::LOAD, CV>;
    auto kernel = leaf_tma_kernel<C, T::S, T::LOAD, CV, MODE>;
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
    if (!encode) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled unavailable");
    CUtensorMap tmap;
    cuuint64_t gdim[2] = {256, static_cast<cuuint64_t>(a.n_full)};
    cuuint64_t gstride[1] = {1024};
    // box = one warp's rows, LOAD bytes of each: exactly one stage (kStageBytes)
    cuuint32_t box[2] = {static_cast<cuuint32_t>(T::LOAD / 4), Cfg::kRowsPerCopy};
    static_assert(Cfg::kStageBytes == Cfg::kRowsPerCopy * T::LOAD, "box and stage size must agree");
    cuuint32_t estride[2] = {1, 1};
    CUresult cr = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t *>(a.in), gdim, gstride,
                         box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         T::LOAD == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
    int bps = 0;
    b3g_status st = kernel_blocks_per_sm(reinterpret_cast<const void *>(kernel), Cfg::kThreads, Cfg::kSmemBytes, dev, bps);
    if (st != B3G_OK) return st;
    const uint64_t grid = grid_for(a.n_tiles, bps, info.sm_count);
    cudaError_t e = launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(Cfg::kThreads), Cfg::kSmemBytes,
                               stream, tmap, a);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "leaf_tma_kernel launch");
}

template <int C, bool CV, uint32_t MODE, bool MIS>
b3g_status launch_async(const LeafArgs &a, cudaStream_t stream, int dev, const DeviceInfo &info) {
    constexpr int S = AsyncTuning<C>::S;
    constexpr size_t smem = AsyncCfg<C, S, MIS>::kSmemBytes;
    auto kernel = leaf_async_kernel<C, S, CV, MODE, MIS>;
    int bps = 0;
    b3g_status st = kernel_blocks_per_sm(reinterpret_cast<const void *>(kernel), C + 32, smem, dev, bps);
    if (st != B3G_OK) return st;
    const uint64_t grid = grid_for(a.n_tiles, bps, info.sm_count);
    cudaError_t e = launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(C + 32), smem, stream, a);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "leaf_async_kernel launch");
}

// Which leaf kernel takes an input with at least one full chunk: a 16-byte aligned base
// goes to the staging that B3G_STAGING selects, any other base to the asynchronous-copy
// kernel, which shifts the blocks out of the aligned-down 16-byte units (a tensor map
// needs an aligned base).  Inputs without a full chunk take the plain-load kernel.
enum class LeafPath { kDirect, kStaged, kStagedMisaligned };

template <int C, bool CV, uint32_t MODE>
b3g_status launch_staged(const LeafArgs &a, LeafPath path, cudaStream_t stream, int dev, const DeviceInfo &info) {
    if (path == LeafPath::kStagedMisaligned) return launch_async<C, CV, MODE, true>(a, stream, dev, info);
#if B3G_STAGING
    return launch_async<C, CV, MODE, false>(a, stream, dev, info);
#else
    return launch_tma<C, CV, MODE>(a, stream, dev, info);
#endif
}

template <int C, bool CV, uint32_t MODE>
b3g_status launch_direct(const LeafArgs &a, cudaStream_t stream, int dev, const DeviceInfo &info) {
    auto kernel = leaf_direct_kernel<C, CV, MODE>;
    int bps = 0;
    b3g_status st = kernel_blocks_per_sm(reinterpret_cast<const void *>(kernel), C, 0, dev, bps);
    if (st != B3G_OK) return st;
    const uint64_t grid = grid_for(a.n_tiles, bps, info.sm_count);
    cudaError_t e = launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(C), 0, stream, a);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "leaf_direct_kernel launch");
}

// The hash mode is a template parameter of the kernels, so that the keyed kernels
// compile exactly as without a mode; chunk CVs exist in keyed mode only.
template <int C>
b3g_status launch_c(const LeafArgs &a, bool chunk_cvs, LeafPath path, cudaStream_t stream, int dev,
                    const DeviceInfo &info) {
    const bool staged = path != LeafPath::kDirect;
    if (a.mode_flags == kModeDefault) {
        if (chunk_cvs) return B3G_ERR_ARG;
        return staged ? launch_staged<C, false, kModeDefault>(a, path, stream, dev, info)
                      : launch_direct<C, false, kModeDefault>(a, stream, dev, info);
    }
    if (a.mode_flags != kModeKeyed) return B3G_ERR_ARG;
    if (staged)
        return chunk_cvs ? launch_staged<C, true, kModeKeyed>(a, path, stream, dev, info)
                         : launch_staged<C, false, kModeKeyed>(a, path, stream, dev, info);
    return chunk_cvs ? launch_direct<C, true, kModeKeyed>(a, stream, dev, info)
                     : launch_direct<C, false, kModeKeyed>(a, stream, dev, info);
}

}  // namespace

const char *kernel_config() {
    static char buf[160];
    static std::once_flag once;
    std::call_once(once, [] {
#if B3G_STAGING
        std::snprintf(buf, sizeof buf,
                      "leaf_async_kernel<%d,%d> min_blocks=%d g_form=%d top_batch=%d pair_noinline=%d grab_block=%d "
                      "wait_hint_ns=%d rot_fma=0x%x pdl=1 modes=2",
                      1 << kDefaultLeavesLog2, AsyncTuning<(1 << kDefaultLeavesLog2)>::S, B3G_ASYNC_MIN_BLOCKS,
                      B3G_G_FORM, B3G_TOP_BATCH, B3G_PAIR_NOINLINE,
                      B3G_GRAB_BLOCK < 0 ? 16 - AsyncTuning<(1 << kDefaultLeavesLog2)>::S : B3G_GRAB_BLOCK,
                      B3G_WAIT_HINT_NS,
                      static_cast<unsigned>(B3G_ROT_FMA));
#else
        std::snprintf(buf, sizeof buf,
                      "leaf_tma_kernel<%d,%d,%d> unroll=%d min_blocks=%d g_form=%d top_batch=%d pair_noinline=%d "
                      "rot_fma=0x%x pdl=1 modes=2",
                      1 << kDefaultLeavesLog2, Tuning<(1 << kDefaultLeavesLog2)>::S,
                      Tuning<(1 << kDefaultLeavesLog2)>::LOAD, kCopyLoopUnroll, B3G_MIN_BLOCKS, B3G_G_FORM,
                      B3G_TOP_BATCH, B3G_PAIR_NOINLINE, static_cast<unsigned>(B3G_ROT_FMA));
#endif
    });
    return buf;
}

bool leaf_takes_tile_counter(const void *in, uint64_t n_full) {
    const bool full = n_full >= 1 && n_full + 256 < (1ull << 31);
    const bool aligned = (reinterpret_cast<uintptr_t>(in) & 15u) == 0;
    return full && (B3G_STAGING || !aligned);
}

b3g_status launch_leaf(const LeafArgs &a, int leaves_log2, bool chunk_cvs, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    DeviceInfo info;
    b3g_status st = device_info(dev, info);
    if (st != B3G_OK) return st;
    // Staged kernels need at least one full chunk (and, for the tensor map, row
    // coordinates that fit in int32); the bulk-tensor-copy kernel also a 16-byte aligned
    // base.
    const bool full = a.n_full >= 1 && a.n_full + 256 < (1ull << 31);
    const bool aligned = (reinterpret_cast<uintptr_t>(a.in) & 15u) == 0;
    const LeafPath path = !full ? LeafPath::kDirect : aligned ? LeafPath::kStaged : LeafPath::kStagedMisaligned;
    switch (leaves_log2) {
        case 5: return launch_c<32>(a, chunk_cvs, path, stream, dev, info);
        case 6: return launch_c<64>(a, chunk_cvs, path, stream, dev, info);
        case 7: return launch_c<128>(a, chunk_cvs, path, stream, dev, info);
        case 8: return launch_c<256>(a, chunk_cvs, path, stream, dev, info);
        default: return B3G_ERR_ARG;
    }
}

}  // namespace b3g

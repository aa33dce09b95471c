// b3g_noalloc.cu -- blake3_keyed_hash_noalloc: the keyed digest without any device
// memory allocation.
//
// Who needs it: some callers cannot allocate device memory at the moment they want a
// digest.  Typical cases are a process whose device memory is already fully owned by
// another allocator (for example a framework's caching allocator that reserved the
// GPU at start-up), a latency-critical loop that cannot accept the device-wide
// synchronisation cudaMalloc/cudaFree may cause, or a service whose policy forbids
// allocation after initialisation.  blake3_keyed_hash needs a few bytes of temporary
// device memory (one 32-byte CV per CTA subtree) and takes them from the stream-ordered
// allocator; blake3_keyed_hash_ws needs the caller to have allocated them.  This entry
// point instead uses a fixed scratch array that is part of the library's device image:
// it exists on every GPU that loads the library, from module load until process exit.
//
// The kernels are the same leaf and reduction kernels as blake3_keyed_hash; only the
// place the CTA roots are kept differs.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "b3g_internal.h"

namespace b3g {
namespace {

// 131,072 CTA roots (16 GiB of input at 128 chunks per CTA), the reduction levels
// after them (128 CVs with groups of 1024; at most 520 with groups of 64, which serve
// up to 32,768 roots) and, in the last 16 bytes, the leaf kernel's tile counter.
constexpr size_t kNoAllocScratchBytes = (4u << 20) + 8192;
constexpr size_t kNoAllocCounterOffset = kNoAllocScratchBytes - 16;
// Inputs above 2^16 chunks (64 MiB) use 128 chunks per CTA subtree, as the one-shot
// digest does: the scratch size above is computed for it.  Smaller inputs use the
// one-shot digest's subtree size (down to 32 chunks, so that every SM gets a CTA), at
// most 2048 roots.
constexpr int kNoAllocLeavesLog2 = kDefaultLeavesLog2;
constexpr uint64_t kNoAllocSmallChunks = 1ull << 16;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device.  Host code cannot use
// the symbol itself (on the host it is only a stand-in), so the address is looked up
// once per device, with that device current, and cached.
b3g_status scratch_address(uint8_t **out) {
    static std::mutex mu;
    static uint8_t *cache[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return B3G_ERR_ARG;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        uint8_t *p = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
        cache[dev] = p;
    }
    *out = cache[dev];
    return B3G_OK;
}

uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
size_t round16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

}  // namespace
}  // namespace b3g

using namespace b3g;

extern "C" b3g_status blake3_keyed_hash_noalloc(const void *d_in, uint64_t len, const uint8_t key[32],
                                                uint8_t *d_out32, b3g_stream_t stream) {
    if (!key || !d_out32 || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(d_out32) & 15u) return B3G_ERR_ALIGN;
    if (len > B3G_NOALLOC_MAX_LEN) return B3G_ERR_WORKSPACE;

    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint64_t n_chunks = len == 0 ? 1 : ceil_div(len, kChunkBytes);
    const int t = n_chunks <= kNoAllocSmallChunks ? leaves_log2_for(n_chunks) : kNoAllocLeavesLog2;
    const uint64_t tiles = ceil_div(n_chunks, 1ull << t);
    const uint64_t group = 1ull << reduce_group_log2(tiles);

    // scratch layout: the CTA roots, then one buffer per further reduction level; the
    // tile counter at its end
    size_t need = tiles > 1 ? round16(tiles * 32) : 0;
    for (uint64_t c = tiles; c > group;) {
        c = ceil_div(c, group);
        need += round16(c * 32);
    }
    if (need > kNoAllocCounterOffset) return B3G_ERR_WORKSPACE;

    uint32_t *status = nullptr;
    b3g_status st = device_status_word(&status);
    if (st != B3G_OK) return st;
    uint8_t *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != B3G_OK) return st;

    LeafArgs a;
    a.in = static_cast<const uint8_t *>(d_in);
    a.len = len;
    a.n_chunks = n_chunks;
    a.n_full = len / kChunkBytes;
    a.counter_base = 0;
    a.n_tiles = tiles;
    a.status = status;
    a.wait_limit_ns = kWaitLimitNs;
    for (int i = 0; i < 8; ++i)
        a.key[i] = static_cast<uint32_t>(key[4 * i]) | (static_cast<uint32_t>(key[4 * i + 1]) << 8) |
                   (static_cast<uint32_t>(key[4 * i + 2]) << 16) | (static_cast<uint32_t>(key[4 * i + 3]) << 24);
    a.mode_flags = kModeKeyed;
    a.root = 1;
    a.tail_bytes = static_cast<uint32_t>(len % kChunkBytes);
    a.ticket = nullptr;
    a.final_out = nullptr;
    a.tile_counter = nullptr;
    if (tiles == 1) {
        a.out = d_out32;
        return launch_leaf(a, t, false, s);
    }
    // Every CTA root and every level buffer is written before it is read within this
    // call, so nothing left in the scratch by an earlier call is ever used.  Only the
    // tile counter (more tiles than resident CTAs) is cleared first.
    a.out = scratch;
    if (tiles > kDynamicMinTiles && leaf_takes_tile_counter(d_in, a.n_full)) {
        a.tile_counter = reinterpret_cast<uint32_t *>(scratch + kNoAllocCounterOffset);
        st = launch_zero_word(a.tile_counter, s);
        if (st != B3G_OK) return st;
    }
    st = launch_leaf(a, t, false, s);
    if (st != B3G_OK) return st;
    const uint8_t *cur = scratch;
    uint8_t *next = scratch + round16(tiles * 32);
    uint64_t c = tiles;
    while (true) {
        ReduceArgs ra;
        ra.in = cur;
        ra.count = c;
        const uint64_t groups = ceil_div(c, group);
        ra.out = groups == 1 ? d_out32 : next;
        std::memcpy(ra.key, a.key, sizeof ra.key);
        ra.mode_flags = kModeKeyed;
        ra.root = 1;
        ra.group = static_cast<uint32_t>(group);
        st = launch_reduce(ra, s);
        if (st != B3G_OK || groups == 1) return st;
        cur = next;
        next += round16(groups * 32);
        c = groups;
    }
}

// b3g_api.cu -- the C ABI of libb3g.so (declared in include/blake3_gb300.h).
//
// Host-side planning only: argument checks, the chunk/tile arithmetic, workspace
// layout and the kernel launches.  All hashing runs on the GPU.
//
// Call structure (source page "BLAKE3 GPU 400x faster hashing", sections
// "我们的实现", "Kernel 1", "Kernel 2 和 3"):
//   1. leaf kernel: chunk CVs and the fused CTA subtree -> one CV per tile of 2^t
//      chunks (or the digest itself when the input fits one tile);
//   2. reduction kernel, relaunched on its own output until one CV remains; the
//      launch with a single group sets ROOT.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "b3g_internal.h"

namespace b3g {

namespace {

thread_local char g_last_cuda_error[256] = "";

// Device status word: bit B3G_DEVICE_STATUS_TIMEOUT is set by a kernel whose
// bounded wait gave up.  One per device (a module-scope variable lives in every
// device's copy of the module).
__device__ uint32_t g_device_status;

constexpr int kMaxDevices = 64;

b3g_status status_word(uint32_t **out) {
    static std::mutex mu;
    static uint32_t *cache[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return B3G_ERR_ARG;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        cache[dev] = static_cast<uint32_t *>(p);
    }
    *out = cache[dev];
    return B3G_OK;
}

uint64_t n_chunks_of(uint64_t len) { return len == 0 ? 1 : (len + kChunkBytes - 1) / kChunkBytes; }

uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

void key_words(const uint8_t key[32], uint32_t out[8]) {
    for (int i = 0; i < 8; ++i)
        out[i] = static_cast<uint32_t>(key[4 * i]) | (static_cast<uint32_t>(key[4 * i + 1]) << 8) |
                 (static_cast<uint32_t>(key[4 * i + 2]) << 16) | (static_cast<uint32_t>(key[4 * i + 3]) << 24);
}

bool valid_leaves_log2(int t) { return t >= kMinLeavesLog2 && t <= kMaxLeavesLog2; }

// Outputs and CV inputs are moved with 16-byte vector accesses.
bool misaligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

size_t round16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// Bytes for the intermediate levels of a reduction of `count` CVs with groups of
// 2^g: every level except the last (which writes the final output) needs a buffer.
size_t reduce_ws(uint64_t count, int g) {
    size_t total = 0;
    uint64_t c = count;
    const uint64_t group = 1ull << g;
    while (c > group) {
        c = ceil_div(c, group);
        total += round16(c * 32);
    }
    return total;
}

// Reduce `count` CVs at d_cvs into d_out32 (see blake3_keyed_reduce_cvs).
b3g_status reduce_levels(const uint8_t *d_cvs, uint64_t count, const uint32_t key[8], uint32_t mode_flags,
                         bool is_root, int g, uint8_t *d_out32, uint8_t *ws, cudaStream_t stream) {
    if (count == 1) {
        cudaError_t e = cudaMemcpyAsync(d_out32, d_cvs, 32, cudaMemcpyDeviceToDevice, stream);
        return e == cudaSuccess ? B3G_OK : cuda_fail(e, "cudaMemcpyAsync");
    }
    const uint64_t group = 1ull << g;
    const uint8_t *cur = d_cvs;
    uint64_t c = count;
    uint8_t *next_buf = ws;
    while (true) {
        ReduceArgs ra;
        ra.in = cur;
        ra.count = c;
        const uint64_t groups = ceil_div(c, group);
        ra.out = groups == 1 ? d_out32 : next_buf;
        std::memcpy(ra.key, key, sizeof ra.key);
        ra.mode_flags = mode_flags;
        ra.root = is_root ? 1u : 0u;
        ra.group = static_cast<uint32_t>(group);
        b3g_status st = launch_reduce(ra, stream);
        if (st != B3G_OK) return st;
        if (groups == 1) return B3G_OK;
        cur = next_buf;
        next_buf += round16(groups * 32);
        c = groups;
    }
}

LeafArgs leaf_args(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                   uint32_t mode_flags, int t, bool root, uint8_t *out, uint32_t *status) {
    LeafArgs a;
    a.in = static_cast<const uint8_t *>(d_in);
    a.len = len;
    a.n_chunks = n_chunks_of(len);
    a.n_full = len / kChunkBytes;
    a.counter_base = chunk_offset;
    a.n_tiles = ceil_div(a.n_chunks, 1ull << t);
    a.out = out;
    a.status = status;
    a.wait_limit_ns = kWaitLimitNs;
    key_words(key, a.key);
    a.mode_flags = mode_flags;
    a.root = root ? 1u : 0u;
    a.tail_bytes = static_cast<uint32_t>(len % kChunkBytes);
    a.ticket = nullptr;
    a.final_out = nullptr;
    a.tile_counter = nullptr;
    return a;
}

// Chunks per CTA subtree (log2) for an input of n chunks.  Large inputs use
// 2^kDefaultLeavesLog2 (128).  For an input of at most 2^16 chunks (64 MiB) with fewer
// than kFullTileMinTiles subtrees of that size, the subtree shrinks (down to 32 chunks)
// until there are at least kSpreadTiles CTAs: each chunk is a chain of 16 dependent
// compressions, so small inputs finish sooner with fewer warps per SM.  From
// kFullTileMinTiles 128-chunk subtrees on (10 MiB), the 128-chunk kernel with at most
// one CTA per SM is faster than the smaller subtrees' kernels (measured on GB300: 10 MiB
// 364 against 330 GB/s, 12 MiB 436 against 391, 16 MiB 579 against 515; at 8 MiB, 64
// subtrees, it is not).  A function of n alone, so that the workspace size is a function
// of the length alone.
constexpr uint64_t kSmallInputChunks = 1ull << 16;
constexpr uint64_t kSpreadTiles = 152;
constexpr uint64_t kFullTileMinTiles = 80;

int choose_leaves_log2(uint64_t n_chunks) {
    int t = kDefaultLeavesLog2;
    if (n_chunks <= kSmallInputChunks && ceil_div(n_chunks, 1ull << t) < kFullTileMinTiles)
        while (t > kMinLeavesLog2 && ceil_div(n_chunks, 1ull << t) < kSpreadTiles) --t;
    return t;
}

// The fused final reduction lives in the bulk-tensor-copy kernel; inputs that take
// the plain-load kernel (misaligned, or no full chunk) use the reduction kernel.
std::atomic<int> g_fused_final{0};

bool fused_path(const void *d_in, uint64_t n_full) {
    return g_fused_final.load(std::memory_order_relaxed) != 0 && n_full >= 1 &&
           (reinterpret_cast<uintptr_t>(d_in) & 15u) == 0;
}

// The whole path: leaf kernel, then the reduction levels.  `ws` must hold
// blake3_workspace_size(len) bytes when more than one tile exists.
// `call_status`: a caller's device word that the kernels of this call report a
// given-up wait in, instead of the per-device status word (NULL: the device word).
b3g_status hash_range(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                      uint32_t mode_flags, bool root, uint8_t *d_out32, uint8_t *ws, cudaStream_t stream,
                      uint32_t *call_status = nullptr) {
    uint32_t *status = call_status;
    b3g_status st = B3G_OK;
    if (!status) st = status_word(&status);
    if (st != B3G_OK) return st;
    const int t = choose_leaves_log2(n_chunks_of(len));
    LeafArgs a = leaf_args(d_in, len, chunk_offset, key, mode_flags, t, root, nullptr, status);
    if (a.n_tiles == 1) {
        a.out = d_out32;
        return launch_leaf(a, t, false, stream);
    }
    a.out = ws;
    if (a.n_tiles <= kMaxFusedTiles && fused_path(d_in, a.n_full)) {
        // few tiles: the last CTA folds the tile CVs itself (one launch, no
        // reduction kernel); its ticket counter sits after the tile CVs
        a.ticket = reinterpret_cast<uint32_t *>(ws + round16(a.n_tiles * 32));
        a.final_out = d_out32;
        st = launch_zero_word(a.ticket, stream);
        if (st != B3G_OK) return st;
        return launch_leaf(a, t, false, stream);
    }
    const int g = reduce_group_log2(a.n_tiles);
    if (a.n_tiles > kDynamicMinTiles && leaf_takes_tile_counter(d_in, a.n_full)) {
        // the tile counter sits after the reduction levels
        a.tile_counter = reinterpret_cast<uint32_t *>(ws + round16(a.n_tiles * 32) + reduce_ws(a.n_tiles, g));
        st = launch_zero_word(a.tile_counter, stream);
        if (st != B3G_OK) return st;
    }
    st = launch_leaf(a, t, false, stream);
    if (st != B3G_OK) return st;
    return reduce_levels(ws, a.n_tiles, a.key, mode_flags, root, g, d_out32, ws + round16(a.n_tiles * 32),
                         stream);
}

size_t hash_workspace(uint64_t len) {
    const uint64_t n = n_chunks_of(len);
    const uint64_t tiles = ceil_div(n, 1ull << choose_leaves_log2(n));
    if (tiles == 1) return 0;
    // the fused path needs 16 bytes for its ticket counter instead of reduction levels;
    // inputs of more than kDynamicMinTiles tiles 16 bytes for a tile counter
    const size_t levels = reduce_ws(tiles, reduce_group_log2(tiles));
    return round16(tiles * 32) + (tiles <= kMaxFusedTiles && levels < 16 ? 16 : levels) +
           (tiles > kDynamicMinTiles ? 16 : 0);
}

// Runs hash_range with a stream-ordered temporary workspace.
b3g_status hash_range_alloc(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                            uint32_t mode_flags, bool root, uint8_t *d_out32, cudaStream_t stream,
                            uint32_t *call_status = nullptr) {
    const size_t need = hash_workspace(len);
    void *ws = nullptr;
    if (need) {
        cudaError_t e = alloc_async(&ws, need, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync");
    }
    b3g_status st = hash_range(d_in, len, chunk_offset, key, mode_flags, root, d_out32, static_cast<uint8_t *>(ws),
                               stream, call_status);
    if (ws) {
        cudaError_t e = cudaFreeAsync(ws, stream);
        if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "cudaFreeAsync");
    }
    return st;
}

}  // namespace

b3g_status device_status_word(uint32_t **out) { return status_word(out); }

int leaves_log2_for(uint64_t n_chunks) { return choose_leaves_log2(n_chunks); }

b3g_status hash_range_ws(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                         uint32_t mode_flags, bool root, uint8_t *d_out32, uint8_t *ws, cudaStream_t stream) {
    return hash_range(d_in, len, chunk_offset, key, mode_flags, root, d_out32, ws, stream);
}

b3g_status reduce_cvs_ws(const uint8_t *d_cvs, uint64_t count, const uint32_t key[8], uint32_t mode_flags,
                         bool root, uint8_t *d_out32, uint8_t *ws, size_t ws_bytes, cudaStream_t stream) {
    if (count == 0 || (count == 1 && root)) return B3G_ERR_ARG;
    const int g = reduce_group_log2(count);
    if (ws_bytes < reduce_ws(count, g)) return B3G_ERR_WORKSPACE;
    return reduce_levels(d_cvs, count, key, mode_flags, root, g, d_out32, ws, stream);
}

namespace {
// > 0: the g_fail_alloc-th next device allocation fails (then the hook is off)
std::atomic<int64_t> g_fail_alloc{0};

bool injected_failure() {
    int64_t v = g_fail_alloc.load(std::memory_order_relaxed);
    while (v > 0)
        if (g_fail_alloc.compare_exchange_weak(v, v - 1, std::memory_order_relaxed)) return v == 1;
    return false;
}
}  // namespace

namespace {
std::atomic<int> g_stream_unbatched{0};
}  // namespace

bool stream_unbatched() { return g_stream_unbatched.load(std::memory_order_relaxed) != 0; }

cudaError_t alloc_async(void **p, size_t bytes, cudaStream_t stream) {
    if (injected_failure()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMallocAsync(p, bytes, stream);
}

cudaError_t alloc_sync(void **p, size_t bytes) {
    if (injected_failure()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}

b3g_status cuda_fail(cudaError_t err, const char *what) {
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s (%d)", what, cudaGetErrorString(err),
                  static_cast<int>(err));
    return B3G_ERR_CUDA;
}

}  // namespace b3g

using namespace b3g;

extern "C" {

const char *blake3_strerror(b3g_status s) {
    switch (s) {
        case B3G_OK: return "success";
        case B3G_ERR_NULL: return "a required pointer is NULL";
        case B3G_ERR_ALIGN: return "misaligned argument (chunk_offset, workspace or a 16-byte aligned pointer)";
        case B3G_ERR_WORKSPACE: return "workspace too small";
        case B3G_ERR_CUDA: return "CUDA runtime error";
        case B3G_ERR_TIMEOUT: return "a device-side bounded wait gave up";
        case B3G_ERR_ARG: return "argument out of range";
    }
    return "unknown status";
}

const char *blake3_last_cuda_error(void) { return g_last_cuda_error; }

int blake3_default_leaves_log2(void) { return kDefaultLeavesLog2; }

const char *blake3_kernel_config(void) { return kernel_config(); }

b3g_status blake3_set_option(b3g_option option, int64_t value) {
    switch (option) {
        case B3G_OPT_FUSED_FINAL:
            g_fused_final.store(value != 0 ? 1 : 0, std::memory_order_relaxed);
            return B3G_OK;
        case B3G_OPT_FAIL_ALLOC:
            if (value < 0) return B3G_ERR_ARG;
            g_fail_alloc.store(value, std::memory_order_relaxed);
            return B3G_OK;
        case B3G_OPT_STREAM_UNBATCHED:
            g_stream_unbatched.store(value != 0 ? 1 : 0, std::memory_order_relaxed);
            return B3G_OK;
    }
    return B3G_ERR_ARG;
}

size_t blake3_workspace_size(uint64_t len) { return hash_workspace(len); }

b3g_status blake3_keyed_hash(const void *d_in, uint64_t len, const uint8_t key[32], uint8_t *d_out32,
                             b3g_stream_t stream) {
    if (!key || !d_out32 || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (misaligned16(d_out32)) return B3G_ERR_ALIGN;
    return hash_range_alloc(d_in, len, 0, key, kModeKeyed, true, d_out32, reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_keyed_hash_ws(const void *d_in, uint64_t len, const uint8_t key[32], uint8_t *d_out32,
                                void *d_ws, size_t ws_bytes, b3g_stream_t stream) {
    if (!key || !d_out32 || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (misaligned16(d_out32)) return B3G_ERR_ALIGN;
    const size_t need = hash_workspace(len);
    if (need) {
        if (!d_ws || ws_bytes < need) return B3G_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(d_ws) & 15u) return B3G_ERR_ALIGN;
    }
    return hash_range(d_in, len, 0, key, kModeKeyed, true, d_out32, static_cast<uint8_t *>(d_ws),
                      reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_keyed_hash_ex(const void *d_in, uint64_t len, const uint8_t key[32], uint8_t *d_out32,
                                void *d_ws, size_t ws_bytes, uint32_t *d_status, b3g_stream_t stream) {
    if (!key || !d_out32 || !d_status || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (misaligned16(d_out32) || (reinterpret_cast<uintptr_t>(d_status) & 3u)) return B3G_ERR_ALIGN;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!d_ws) return hash_range_alloc(d_in, len, 0, key, kModeKeyed, true, d_out32, s, d_status);
    const size_t need = hash_workspace(len);
    if (need) {
        if (ws_bytes < need) return B3G_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(d_ws) & 15u) return B3G_ERR_ALIGN;
    }
    return hash_range(d_in, len, 0, key, kModeKeyed, true, d_out32, static_cast<uint8_t *>(d_ws), s, d_status);
}

b3g_status blake3_hash(const void *d_in, uint64_t len, uint8_t *d_out32, b3g_stream_t stream) {
    if (!d_out32 || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (misaligned16(d_out32)) return B3G_ERR_ALIGN;
    uint8_t iv[32];
    iv_key_bytes(iv);
    return hash_range_alloc(d_in, len, 0, iv, kModeDefault, true, d_out32, reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_hash_ws(const void *d_in, uint64_t len, uint8_t *d_out32, void *d_ws, size_t ws_bytes,
                          b3g_stream_t stream) {
    if (!d_out32 || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (misaligned16(d_out32)) return B3G_ERR_ALIGN;
    const size_t need = hash_workspace(len);
    if (need) {
        if (!d_ws || ws_bytes < need) return B3G_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(d_ws) & 15u) return B3G_ERR_ALIGN;
    }
    uint8_t iv[32];
    iv_key_bytes(iv);
    return hash_range(d_in, len, 0, iv, kModeDefault, true, d_out32, static_cast<uint8_t *>(d_ws),
                      reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_keyed_chunk_cvs(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                                  uint8_t *d_cvs, b3g_stream_t stream) {
    if (!key || !d_cvs || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (misaligned16(d_cvs)) return B3G_ERR_ALIGN;
    uint32_t *status = nullptr;
    b3g_status st = status_word(&status);
    if (st != B3G_OK) return st;
    LeafArgs a = leaf_args(d_in, len, chunk_offset, key, kModeKeyed, kDefaultLeavesLog2, false, d_cvs, status);
    return launch_leaf(a, kDefaultLeavesLog2, true, reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_keyed_subtree_root(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                                     int is_root, uint8_t *d_out32, b3g_stream_t stream) {
    if (!key || !d_out32 || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (misaligned16(d_out32)) return B3G_ERR_ALIGN;
    const uint64_t n = n_chunks_of(len);
    uint64_t p = 1;
    while (p < n) p <<= 1;
    if (chunk_offset % p != 0) return B3G_ERR_ALIGN;
    return hash_range_alloc(d_in, len, chunk_offset, key, kModeKeyed, is_root != 0, d_out32,
                            reinterpret_cast<cudaStream_t>(stream));
}

uint64_t blake3_tile_count(uint64_t len, int leaves_log2) {
    if (leaves_log2 == -1) leaves_log2 = kDefaultLeavesLog2;
    if (!valid_leaves_log2(leaves_log2)) return 0;
    return ceil_div(n_chunks_of(len), 1ull << leaves_log2);
}

b3g_status blake3_keyed_tile_roots_ex(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                                      int leaves_log2, int is_root, uint8_t *d_roots, uint32_t *d_tile_counter,
                                      b3g_stream_t stream) {
    if (!key || !d_roots || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (misaligned16(d_roots) || (reinterpret_cast<uintptr_t>(d_tile_counter) & 3u)) return B3G_ERR_ALIGN;
    if (leaves_log2 == -1) leaves_log2 = kDefaultLeavesLog2;
    if (!valid_leaves_log2(leaves_log2)) return B3G_ERR_ARG;
    uint32_t *status = nullptr;
    b3g_status st = status_word(&status);
    if (st != B3G_OK) return st;
    LeafArgs a = leaf_args(d_in, len, chunk_offset, key, kModeKeyed, leaves_log2, is_root != 0, d_roots, status);
    a.tile_counter = d_tile_counter;
    return launch_leaf(a, leaves_log2, false, reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_keyed_tile_roots(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                                   int leaves_log2, int is_root, uint8_t *d_roots, b3g_stream_t stream) {
    return blake3_keyed_tile_roots_ex(d_in, len, chunk_offset, key, leaves_log2, is_root, d_roots, nullptr, stream);
}

size_t blake3_reduce_workspace_size(uint64_t count, int group_log2) {
    if (group_log2 == -1) group_log2 = reduce_group_log2(count);
    if (group_log2 < 1 || group_log2 > kMaxGroupLog2 || count == 0) return 0;
    return reduce_ws(count, group_log2);
}

b3g_status blake3_keyed_reduce_cvs(const uint8_t *d_cvs, uint64_t count, const uint8_t key[32], int is_root,
                                   int group_log2, uint8_t *d_out32, void *d_ws, size_t ws_bytes,
                                   b3g_stream_t stream) {
    if (!key || !d_cvs || !d_out32) return B3G_ERR_NULL;
    if (misaligned16(d_cvs) || misaligned16(d_out32)) return B3G_ERR_ALIGN;
    if (group_log2 == -1) group_log2 = reduce_group_log2(count);
    if (count == 0 || group_log2 < 1 || group_log2 > kMaxGroupLog2) return B3G_ERR_ARG;
    if (count == 1 && is_root) return B3G_ERR_ARG;
    const size_t need = reduce_ws(count, group_log2);
    if (need) {
        if (!d_ws || ws_bytes < need) return B3G_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(d_ws) & 15u) return B3G_ERR_ALIGN;
    }
    uint32_t kw[8];
    key_words(key, kw);
    return reduce_levels(d_cvs, count, kw, kModeKeyed, is_root != 0, group_log2, d_out32,
                         static_cast<uint8_t *>(d_ws), reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_device_status(uint32_t *status_out) {
    if (!status_out) return B3G_ERR_NULL;
    uint32_t *status = nullptr;
    b3g_status st = status_word(&status);
    if (st != B3G_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    uint32_t v = 0;
    e = cudaMemcpy(&v, status, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
    e = cudaMemset(status, 0, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    *status_out = v;
    return B3G_OK;
}

b3g_status blake3_selftest_bounded_wait(uint32_t limit_us, int *timed_out_out) {
    if (!timed_out_out) return B3G_ERR_NULL;
    if (limit_us < 1 || limit_us > 10000000u) return B3G_ERR_ARG;
    int *d_flag = nullptr;
    cudaError_t e = alloc_sync(reinterpret_cast<void **>(&d_flag), sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    b3g_status st = launch_wait_probe(static_cast<uint64_t>(limit_us) * 1000ull, d_flag, nullptr);
    int h = -1;
    if (st == B3G_OK) {
        e = cudaMemcpy(&h, d_flag, sizeof h, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) st = cuda_fail(e, "cudaMemcpy(flag)");
    }
    cudaFree(d_flag);
    if (st == B3G_OK) *timed_out_out = h;
    return st;
}

b3g_status blake3_selftest_bounded_wait_ex(uint32_t limit_us, uint32_t *d_status, b3g_stream_t stream) {
    if (!d_status) return B3G_ERR_NULL;
    if (limit_us < 1 || limit_us > 10000000u) return B3G_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(d_status) & 3u) return B3G_ERR_ALIGN;
    return launch_wait_probe_status(static_cast<uint64_t>(limit_us) * 1000ull, d_status,
                                    reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_selftest_compress_latency(int lanes_per_chunk, uint32_t chain, const uint8_t key[32],
                                            uint8_t *d_cvs, uint64_t *d_cycles, b3g_stream_t stream) {
    if (!key || !d_cvs || !d_cycles) return B3G_ERR_NULL;
    if ((lanes_per_chunk != 1 && lanes_per_chunk != 4) || chain < 1 || chain > (1u << 20)) return B3G_ERR_ARG;
    if (misaligned16(d_cvs) || (reinterpret_cast<uintptr_t>(d_cycles) & 7u)) return B3G_ERR_ALIGN;
    LatencyArgs a;
    key_words(key, a.key);
    a.out = d_cvs;
    a.cycles = reinterpret_cast<unsigned long long *>(d_cycles);
    return launch_compress_latency(lanes_per_chunk, chain, a, reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_selftest_compress_rate(uint32_t blocks, uint32_t iters, uint32_t *d_sink, b3g_stream_t stream) {
    if (!d_sink) return B3G_ERR_NULL;
    if (blocks < 1 || blocks > (1u << 20) || iters < 1 || iters > (1u << 20)) return B3G_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(d_sink) & 3u) return B3G_ERR_ALIGN;
    return launch_compress_rate(blocks, iters, d_sink, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// b3g_internal.h -- launch-level interface between the C ABI (b3g_api.cu) and the
// kernel translation units (b3g_leaf.cu, b3g_reduce.cu).  Not installed.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/blake3_gb300.h"

namespace b3g {

constexpr uint64_t kChunkBytes = 1024;
constexpr int kMinLeavesLog2 = 5;
constexpr int kMaxLeavesLog2 = 8;
constexpr int kDefaultLeavesLog2 = 7;  // 128 chunks per CTA (measured best on GB300)
constexpr int kMaxGroupLog2 = 10;
constexpr int kDefaultGroupLog2 = 10;
// Group size (log2) of a root reduction of `count` CVs when the caller does not fix
// it.  The reduction is a chain of ceil(log2(count)) dependent compressions whatever
// the grouping; what the grouping changes is the launch count and whether a level
// crowds one SM.  Groups of 1024 put 16 warps of parents on one SM at the first
// level, 4 per scheduler, so that level runs at throughput instead of latency;
// groups of 64 are one warp each.  Measured from CUDA graphs on GB300: 2048 CVs
// 11.5 -> 8.8 us, 32,768 CVs 14.1 -> 12.7 us with groups of 64; above that the third
// launch of the small groups costs more (98,305 CVs: 17.2 us with 1024, 19.6 with 64).
constexpr uint64_t kSmallGroupMaxCount = 1ull << 15;
constexpr int kSmallGroupLog2 = 6;
inline int reduce_group_log2(uint64_t count) {
    return count <= kSmallGroupMaxCount ? kSmallGroupLog2 : kDefaultGroupLog2;
}
// Default limit of every device-side wait: far above any real wait (microseconds),
// far below a hang.
constexpr uint32_t kWaitLimitNs = 2000000000u;

// Hash modes (page section "BLAKE3": the initial chaining value is an IV by default,
// the user's key in keyed mode).  A mode is its initial CV (the key words, or the IV)
// and the flag bits every one of its compressions carries.
constexpr uint32_t kModeKeyed = 16u;   // KEYED_HASH
constexpr uint32_t kModeDefault = 0u;  // no mode bit
constexpr uint32_t kIvWords[8] = {0x6A09E667u, 0xBB67AE85u, 0x3C6EF372u, 0xA54FF53Au,
                                  0x510E527Fu, 0x9B05688Cu, 0x1F83D9ABu, 0x5BE0CD19u};

// The IV as 32 little-endian key bytes: the default mode runs the keyed machinery
// with these as its key and kModeDefault as its flag bits.
inline void iv_key_bytes(uint8_t out[32]) {
    for (int i = 0; i < 8; ++i)
        for (int b = 0; b < 4; ++b) out[4 * i + b] = static_cast<uint8_t>(kIvWords[i] >> (8 * b));
}

// Arguments of the leaf kernels (page section "Kernel 1": every CTA compresses a
// group of 2^t chunks and reduces them to one subtree CV).
struct LeafArgs {
    const uint8_t *in;      // device bytes
    uint64_t len;           // bytes
    uint64_t n_chunks;      // max(1, ceil(len / 1024))
    uint64_t n_full;        // len / 1024: chunks that are complete
    uint64_t counter_base;  // global index of the first chunk
    uint64_t n_tiles;       // ceil(n_chunks / 2^t)
    uint8_t *out;           // tile CVs (32 B each) or chunk CVs (32 B each)
    uint32_t *status;       // device status word
    uint32_t wait_limit_ns; // limit of every device-side wait (at most 4.29 s)
    uint32_t mode_flags;    // flag bits of the hash mode on every compression
    uint32_t key[8];        // initial CV of every chunk and parent (the key, or the IV)
    uint32_t root;        // ROOT on the final compression if the whole tree is one tile
    uint32_t tail_bytes;  // bytes of the partial last chunk; 0 if none
    // Fused final reduction (at most 32 tiles): when `ticket` is not NULL (a zeroed
    // counter), the reducer that finishes the last tile folds all tile CVs (in `out`)
    // to the root, with ROOT when `root` is set, and writes it to `final_out`.
    uint32_t *ticket;
    uint8_t *final_out;
    // Dynamic tile scheduling (asynchronous-copy kernel only): a zeroed counter from
    // which the CTAs take their tiles after the first (NULL: tiles blockIdx.x + i gridDim.x).
    uint32_t *tile_counter;
};

// Inputs with more tiles than this take their tiles from a counter (the CTA count of a
// 128-chunk launch is 5 per SM, 760 on GB300: below it every CTA has one tile).
constexpr uint64_t kDynamicMinTiles = 760;

// Whether launch_leaf would run a kernel that takes tiles from LeafArgs::tile_counter
// for an input at `in` with `n_full` full chunks.
bool leaf_takes_tile_counter(const void *in, uint64_t n_full);

// Largest tile count the fused final reduction handles (one CV per lane of a warp).
constexpr uint64_t kMaxFusedTiles = 32;

// Arguments of the CV reduction kernel (page section "Kernel 2 和 3").
struct ReduceArgs {
    const uint8_t *in;  // count CVs
    uint64_t count;
    uint8_t *out;       // ceil(count / group) CVs
    uint32_t key[8];
    uint32_t mode_flags;
    uint32_t root;      // ROOT on the final compression when one group remains
    uint32_t group;     // CVs per CTA, a power of two in 2..1024
};

// Launches the leaf kernel: per tile CVs (chunk_cvs == false) or per chunk CVs.
// Chooses the bulk-tensor-copy path when `in` is 16-byte aligned and holds at
// least one full chunk, the plain-load path otherwise.
b3g_status launch_leaf(const LeafArgs &args, int leaves_log2, bool chunk_cvs, cudaStream_t stream);

// "leaf_tma_kernel<C,S,LOAD> unroll=.. min_blocks=.. g_form=.." of the default tile size.
const char *kernel_config();

// One level of CV reduction.
b3g_status launch_reduce(const ReduceArgs &args, cudaStream_t stream);

// Zeroes one device word in stream order (a one-thread kernel launched with
// programmatic stream serialization, so that the launch behind it overlaps it).
b3g_status launch_zero_word(uint32_t *p, cudaStream_t stream);

// One-thread bounded-wait probe; writes 1 to *d_flag if the wait gave up.
b3g_status launch_wait_probe(uint64_t limit_ns, int *d_flag, cudaStream_t stream);
// The same probe, ORing B3G_DEVICE_STATUS_TIMEOUT into *d_status (stream ordered) if the wait gave up.
b3g_status launch_wait_probe_status(uint64_t limit_ns, uint32_t *d_status, cudaStream_t stream);
// `blocks` CTAs of 128 threads, each thread `iters` chained compressions, no memory traffic
b3g_status launch_compress_rate(uint32_t blocks, uint32_t iters, uint32_t *d_sink, cudaStream_t stream);

// Arguments of the compression-latency self-test (several lanes per chunk).
struct LatencyArgs {
    uint32_t key[8];
    uint8_t *out;                // 32 / lanes CVs of 32 bytes
    unsigned long long *cycles;  // clock cycles of the whole chain (lane 0)
};
// One warp: chains of `chain` dependent compressions with 1 or 4 lanes per chain.
b3g_status launch_compress_latency(int lanes, uint32_t chain, const LatencyArgs &a, cudaStream_t stream);

// Records a CUDA error for blake3_last_cuda_error() and returns B3G_ERR_CUDA.
b3g_status cuda_fail(cudaError_t err, const char *what);

// Every device allocation of the library: stream-ordered, and plain.  Both return
// cudaErrorMemoryAllocation without allocating when the failure hook
// (B3G_OPT_FAIL_ALLOC) selects this allocation.
cudaError_t alloc_async(void **p, size_t bytes, cudaStream_t stream);
cudaError_t alloc_sync(void **p, size_t bytes);

// B3G_OPT_STREAM_UNBATCHED: the streaming hasher's one-piece-at-a-time path is forced.
bool stream_unbatched();

// Launch with programmatic stream serialization: the grid may start while the grid
// ahead of it in the stream is finishing.  Every kernel launched this way calls
// grid_dependency_wait() before its first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// CTA subtree size (log2 of the chunks) the one-shot digest uses for n chunks: 128
// chunks, fewer (down to 32) for inputs of at most 2^16 chunks so that at least one
// CTA per SM exists.
int leaves_log2_for(uint64_t n_chunks);

// Device address of the current device's status word (looked up once per device).
b3g_status device_status_word(uint32_t **out);

// The CV of the subtree made of the chunks of d_in[0..len) whose first chunk has global
// index chunk_offset (ROOT on the final compression if root), written to d_out32;
// ws holds blake3_workspace_size(len) bytes.
b3g_status hash_range_ws(const void *d_in, uint64_t len, uint64_t chunk_offset, const uint8_t key[32],
                         uint32_t mode_flags, bool root, uint8_t *d_out32, uint8_t *ws, cudaStream_t stream);

// Reduction of `count` CVs (a perfect or right-folded subtree) to d_out32 with groups of
// 2^kDefaultGroupLog2; ws holds blake3_reduce_workspace_size(count, -1) bytes.
b3g_status reduce_cvs_ws(const uint8_t *d_cvs, uint64_t count, const uint32_t key[8], uint32_t mode_flags,
                         bool root, uint8_t *d_out32, uint8_t *ws, size_t ws_bytes, cudaStream_t stream);

}  // namespace b3g

/*
 * blake3_gb300.h -- C ABI of libb3g.so: the keyed BLAKE3 digest of one buffer that
 * already sits in GPU memory, computed by hand-written sm_103a (GB300) kernels.
 *
 * What is computed (source page: "BLAKE3 GPU 400x faster hashing", qfminer.top):
 *   - section "BLAKE3": the input is cut into 1024-byte chunks and each chunk into
 *     64-byte blocks; each block is compressed (7 rounds) with the running chaining
 *     value (CV), a per-chunk counter, the block length and flags; the key is the
 *     starting CV (keyed mode, the only mode the page uses); the chunk CVs are then
 *     paired into parent nodes until one CV is left, with a full left subtree of a
 *     power-of-two chunk count that is at least as large as its right sibling.
 *   - section "压缩函数": CHUNK_START on a chunk's first block, CHUNK_END on its last.
 *   - section "Merkle Tree 归约": parents use counter 0, block length 64 and flags
 *     KEYED_HASH|PARENT; non-power-of-two counts fold their binary decomposition
 *     from right to left.
 *   - section "Kernel 2 和 3": ROOT is set on the final compression only.
 *   - section "不完整块的处理": the last chunk (and block) may be partial; it is
 *     zero padded and its block length is its true byte count.
 *   The round constants (IV, G rotations, message permutation, flag bit values)
 *   are those of the published BLAKE3 specification (O'Connor et al., 2020).
 *
 * Conventions shared by every entry point:
 *   - Pointers named d_* are DEVICE pointers on the current CUDA device; `key` is a
 *     HOST pointer to 32 bytes, copied into the launch parameters before the call
 *     returns (it may be freed right after).  Byte strings (key, CVs, digest) are
 *     32 bytes, little-endian words, exactly as BLAKE3 defines them.
 *   - The caller owns every buffer.  Nothing is retained across calls except a
 *     per-device cache of launch settings and the device status word.
 *   - All calls that take a stream are asynchronous on it: no host synchronisation
 *     and no device-to-host copy.  Errors found on the host (arguments, launch)
 *     are returned; errors found on the device (a bounded wait that gave up) are
 *     recorded in the device status word, read by blake3_device_status(), or in a
 *     caller's own status word (blake3_keyed_hash_ex).
 *   - len == 0 is valid (the empty input has one empty chunk); d_in may then be NULL.
 *   - d_in may have any alignment.  A 16-byte aligned d_in with at least one full
 *     chunk takes the bulk-tensor-copy (TMA) path; other inputs take a path with
 *     plain bounds-checked loads.  Both give identical results.
 *   - Device pointers that receive CVs or a digest (d_out32, d_cvs, d_roots), and
 *     the CVs given to blake3_keyed_reduce_cvs, must be 16-byte aligned (they are
 *     moved with 16-byte vector accesses); otherwise the call returns B3G_ERR_ALIGN.
 *   - A call never aborts the process; it returns a b3g_status.
 */
#ifndef BLAKE3_GB300_H
#define BLAKE3_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *b3g_stream_t;

typedef enum {
    B3G_OK = 0,
    B3G_ERR_NULL = 1,      /* a required pointer is NULL */
    B3G_ERR_ALIGN = 2,     /* chunk_offset not a multiple of the subtree's size, or a
                              pointer lacks the 16-byte alignment it needs */
    B3G_ERR_WORKSPACE = 3, /* the workspace given is smaller than required */
    B3G_ERR_CUDA = 4,      /* a CUDA runtime call failed (see blake3_last_cuda_error) */
    B3G_ERR_TIMEOUT = 5,   /* a device-side bounded wait gave up (device status word) */
    B3G_ERR_ARG = 6,       /* an argument is out of range */
} b3g_status;

/* Bit set in the device status word when a kernel's bounded wait gave up. */
#define B3G_DEVICE_STATUS_TIMEOUT 1u

/* Static text for a status code; never NULL. */
const char *blake3_strerror(b3g_status status);

/* Text of the last CUDA error seen by this thread inside the library ("" if none). */
const char *blake3_last_cuda_error(void);

/* Chunks per CTA subtree used when leaves_log2 is -1 (a power of two: 2^7 = 128). */
int blake3_default_leaves_log2(void);

/* Library-wide options (process-wide, thread-safe to set; they apply to calls made
 * after the change). */
typedef enum {
    /* 0 (default) or 1.  With 1, an input of at most 32 CTA subtrees is reduced to its
     * digest by the CTA that finishes last (an atomic ticket counter, zeroed on the
     * stream by a one-thread kernel) instead of by a second kernel launch.  Measured on
     * GB300 it is slower for 1 MiB (22.9 vs 21.0 us per digest in a CUDA graph): the
     * zeroing costs more than the launch it saves.  Applies to 16-byte aligned inputs
     * with at least one full chunk. */
    B3G_OPT_FUSED_FINAL = 1,
    /* Test hook for failure handling (no GPU fault involved): with value n > 0, the n-th
     * next device allocation the library makes fails as if the device were out of memory
     * (the call returns B3G_ERR_CUDA, except a streaming hasher's optional 64 MiB buffer,
     * which is then simply not used); afterwards the hook is off again.  0 turns it off. */
    B3G_OPT_FAIL_ALLOC = 2,
    /* Test hook: 0 (default) or 1.  With 1 the streaming hasher pushes every piece of a
     * run with its own subtree and merge launches instead of the batched launches (the
     * path it otherwise takes only for runs beyond the batch limits). */
    B3G_OPT_STREAM_UNBATCHED = 3,
} b3g_option;

/* Sets an option.  Errors: B3G_ERR_ARG (unknown option). */
b3g_status blake3_set_option(b3g_option option, int64_t value);

/* Static text naming the compiled configuration of the leaf kernel for the default
 * subtree size, e.g. "leaf_tma_kernel<128,3,64> unroll=1 min_blocks=0 g_form=3"
 * (chunks per CTA, stages per consumer warp, bytes per copy, build options). */
const char *blake3_kernel_config(void);

/*
 * blake3_keyed_hash -- the digest of d_in[0..len) under `key`, written to d_out32.
 * Page sections "BLAKE3" (chunking, tree rules), "Kernel 1" (leaf kernel with the
 * fused subtree), "Kernel 2 和 3" (reduction of the subtree roots, ROOT last).
 * Temporary device memory (32 bytes per CTA subtree: per 128 chunks, or per 32..64
 * chunks for inputs of at most 64 MiB) comes from the stream-ordered allocator
 * (cudaMallocAsync/cudaFreeAsync on `stream`).
 * Errors: B3G_ERR_NULL (key or d_out32 NULL, or d_in NULL with len > 0),
 * B3G_ERR_CUDA.
 */
b3g_status blake3_keyed_hash(const void *d_in, uint64_t len, const uint8_t key[32],
                             uint8_t *d_out32, b3g_stream_t stream);

/* Bytes of device workspace blake3_keyed_hash_ws needs for a len-byte input
 * (0 when the input fits one CTA subtree). */
size_t blake3_workspace_size(uint64_t len);

/*
 * blake3_keyed_hash_ws -- as blake3_keyed_hash, with caller-provided device
 * workspace d_ws of ws_bytes bytes (at least blake3_workspace_size(len), 16-byte
 * aligned).  Performs no allocation.  Concurrent calls must not share d_ws.
 * Errors: as blake3_keyed_hash, plus B3G_ERR_WORKSPACE (too small or NULL when
 * needed) and B3G_ERR_ALIGN (d_ws not 16-byte aligned).
 */
b3g_status blake3_keyed_hash_ws(const void *d_in, uint64_t len, const uint8_t key[32],
                                uint8_t *d_out32, void *d_ws, size_t ws_bytes,
                                b3g_stream_t stream);

/*
 * blake3_keyed_hash_ex -- as blake3_keyed_hash_ws (d_ws != NULL) or blake3_keyed_hash
 * (d_ws == NULL: temporary workspace from the stream-ordered allocator), with a
 * per-call status word.  d_status is a 4-byte aligned DEVICE word owned by the caller:
 * a kernel of this call whose bounded wait gives up ORs B3G_DEVICE_STATUS_TIMEOUT into
 * it, in stream order, instead of into the per-device word; the library never clears
 * it.  So the outcome of this one call is known from a 4-byte device-to-host copy on
 * `stream` after it, without synchronising the device or touching other streams' calls
 * (the caller zeroes the word before the call, or keeps ORing several calls into it).
 * With the word clear the digest in d_out32 is valid; with the bit set it is not.
 * It is the failure detection of the leaf and reduction kernels, and has no
 * counterpart in the page.
 * Errors: as blake3_keyed_hash_ws, plus B3G_ERR_NULL (d_status NULL) and
 * B3G_ERR_ALIGN (d_status not 4-byte aligned).
 */
b3g_status blake3_keyed_hash_ex(const void *d_in, uint64_t len, const uint8_t key[32],
                                uint8_t *d_out32, void *d_ws, size_t ws_bytes,
                                uint32_t *d_status, b3g_stream_t stream);

/*
 * blake3_hash / blake3_hash_ws -- the digest in the default (unkeyed) mode.  Page
 * section "BLAKE3": a chunk's first block starts from an IV by default and from the
 * user's key in keyed mode.  Here every chunk and every parent starts from the IV and
 * no compression carries KEYED_HASH (the specification's hash mode); the kernels,
 * tree, workspace size (blake3_workspace_size), alignment rules and errors are those
 * of blake3_keyed_hash / blake3_keyed_hash_ws, without the key argument.
 */
b3g_status blake3_hash(const void *d_in, uint64_t len, uint8_t *d_out32, b3g_stream_t stream);
b3g_status blake3_hash_ws(const void *d_in, uint64_t len, uint8_t *d_out32, void *d_ws, size_t ws_bytes,
                          b3g_stream_t stream);

/*
 * blake3_keyed_chunk_cvs -- the CV of every chunk of d_in[0..len), none with ROOT,
 * chunk i using counter chunk_offset + i (page section "压缩函数": one thread per
 * chunk, 16 chained block compressions).  d_cvs receives max(1, ceil(len/1024))
 * CVs of 32 bytes, in chunk order.
 * Errors: B3G_ERR_NULL, B3G_ERR_CUDA.
 */
b3g_status blake3_keyed_chunk_cvs(const void *d_in, uint64_t len, uint64_t chunk_offset,
                                  const uint8_t key[32], uint8_t *d_cvs, b3g_stream_t stream);

/*
 * blake3_keyed_subtree_root -- the CV of the subtree whose leaves are the chunks of
 * d_in[0..len), the first chunk having global index chunk_offset.  With is_root != 0
 * the final compression carries ROOT (then, with chunk_offset 0, this is the digest).
 * The chunk range must be a subtree of the whole input's tree: chunk_offset must be
 * a multiple of the smallest power of two >= the chunk count, and a partial last
 * chunk or a non-power-of-two count is only valid for the input's last subtree (the
 * caller's responsibility; it cannot be checked here).  Temporary memory as in
 * blake3_keyed_hash.
 * Errors: B3G_ERR_NULL, B3G_ERR_ALIGN (chunk_offset misaligned), B3G_ERR_CUDA.
 */
b3g_status blake3_keyed_subtree_root(const void *d_in, uint64_t len, uint64_t chunk_offset,
                                     const uint8_t key[32], int is_root, uint8_t *d_out32,
                                     b3g_stream_t stream);

/* Number of CTA subtree roots blake3_keyed_tile_roots writes: ceil(chunks / 2^leaves_log2).
 * Returns 0 for a leaves_log2 outside 5..8 (or -1 for the default). */
uint64_t blake3_tile_count(uint64_t len, int leaves_log2);

/*
 * blake3_keyed_tile_roots -- the leaf kernel alone (page section "Kernel 1"): every
 * aligned group of 2^leaves_log2 chunks (leaves_log2 in 5..8, or -1 for the default)
 * is compressed and reduced inside one CTA to its subtree CV; the last group may be
 * smaller and is folded right to left.  d_roots receives blake3_tile_count() CVs.
 * chunk_offset as in blake3_keyed_subtree_root.  If there is a single group and
 * is_root != 0, its CV is the finished digest (ROOT set on the final compression);
 * with several groups is_root is ignored.
 * Errors: B3G_ERR_NULL, B3G_ERR_ARG (leaves_log2), B3G_ERR_CUDA.
 */
b3g_status blake3_keyed_tile_roots(const void *d_in, uint64_t len, uint64_t chunk_offset,
                                   const uint8_t key[32], int leaves_log2, int is_root,
                                   uint8_t *d_roots, b3g_stream_t stream);

/*
 * blake3_keyed_tile_roots_ex -- as blake3_keyed_tile_roots, with dynamic tile
 * scheduling.  d_tile_counter is a 4-byte aligned DEVICE word that the caller has set
 * to zero on `stream` before the call (or NULL: the static order of
 * blake3_keyed_tile_roots).  After its first tile each persistent CTA takes its next
 * tile from the counter, so CTAs that run faster take more tiles and all of them
 * finish together; the warp scheduler favours some CTAs of an SM over others, which
 * leaves a static split with idle warps in its second half.  The roots are the same
 * either way.  The counter is used only by the asynchronous-copy leaf kernel (see
 * blake3_kernel_config); the other kernels ignore it.  One counter serves one call at
 * a time.  A call whose kernels complete without a given-up wait leaves the counter at
 * zero again (the CTAs take from it exactly once per tile, and the last take resets
 * it), so a caller that reuses the counter for calls in stream order clears it once;
 * after a call that reported B3G_DEVICE_STATUS_TIMEOUT it must be cleared again.
 * Scheduling only; the page's Kernel 1 assigns tiles statically.
 * Errors: as blake3_keyed_tile_roots, plus B3G_ERR_ALIGN (d_tile_counter).
 */
b3g_status blake3_keyed_tile_roots_ex(const void *d_in, uint64_t len, uint64_t chunk_offset,
                                      const uint8_t key[32], int leaves_log2, int is_root,
                                      uint8_t *d_roots, uint32_t *d_tile_counter,
                                      b3g_stream_t stream);

/* Device workspace bytes blake3_keyed_reduce_cvs needs for `count` CVs and groups of
 * 2^group_log2 (group_log2 in 1..10, or -1 for the default: 6 for at most 32,768 CVs,
 * else 10). */
size_t blake3_reduce_workspace_size(uint64_t count, int group_log2);

/*
 * blake3_keyed_reduce_cvs -- reduce `count` (>= 1) consecutive subtree CVs d_cvs
 * (the left-to-right leaves of one tree, each an aligned power-of-two subtree except
 * possibly the last) to one CV in d_out32 (page section "Kernel 2 和 3"): each CTA
 * reduces an aligned group of 2^group_log2 CVs, and launches repeat until one CV is
 * left; with is_root != 0 the final compression carries ROOT.  count == 1 copies the
 * CV (is_root must then be 0: ROOT cannot be added to a finished CV).
 * Errors: B3G_ERR_NULL, B3G_ERR_ARG (count 0, group_log2, count 1 with is_root),
 * B3G_ERR_WORKSPACE, B3G_ERR_ALIGN (d_ws not 16-byte aligned), B3G_ERR_CUDA.
 */
b3g_status blake3_keyed_reduce_cvs(const uint8_t *d_cvs, uint64_t count, const uint8_t key[32],
                                   int is_root, int group_log2, uint8_t *d_out32, void *d_ws,
                                   size_t ws_bytes, b3g_stream_t stream);

/*
 * blake3_device_status -- waits for the current device to go idle, stores the device
 * status word (0, or B3G_DEVICE_STATUS_TIMEOUT) in *status_out and clears it.
 * Errors: B3G_ERR_NULL, B3G_ERR_CUDA.
 */
b3g_status blake3_device_status(uint32_t *status_out);

/*
 * blake3_selftest_bounded_wait -- launches one thread that waits on a shared-memory
 * barrier nobody arrives on, with a limit of limit_us microseconds (1..10^7), and
 * stores 1 in *timed_out_out if the wait gave up (the expected outcome), else 0.
 * This exercises the same bounded wait the hashing kernels use, so that the
 * give-up path is tested without a hang.  Synchronous.  Does not touch the status
 * word.  Errors: B3G_ERR_NULL, B3G_ERR_ARG, B3G_ERR_CUDA.
 */
b3g_status blake3_selftest_bounded_wait(uint32_t limit_us, int *timed_out_out);

/*
 * blake3_selftest_bounded_wait_ex -- the same probe, asynchronous on `stream`,
 * reporting like the hashing kernels of blake3_keyed_hash_ex: if its wait gives up
 * (the expected outcome) it ORs B3G_DEVICE_STATUS_TIMEOUT into the caller's 4-byte
 * aligned device word d_status, in stream order.  Errors: B3G_ERR_NULL, B3G_ERR_ARG
 * (limit_us outside 1..10^7), B3G_ERR_ALIGN, B3G_ERR_CUDA.
 */
b3g_status blake3_selftest_bounded_wait_ex(uint32_t limit_us, uint32_t *d_status, b3g_stream_t stream);

/*
 * blake3_selftest_compress_latency -- several threads per chunk (page section
 * "未来工作": threads could share the work of one chunk).  Launches ONE warp on `stream`
 * that runs chains of `chain` (1..2^20) dependent keyed compressions:
 *   lanes_per_chunk = 1: 32 chains, one per lane, with the hashing kernels' compression;
 *   lanes_per_chunk = 4: 8 chains, one per group of 4 lanes, each lane holding one
 *     column of the state (the column step is one G per lane; shuffles rotate the rows
 *     for the diagonal step and back).
 * Chain g starts from the key and compresses, in step j, the 64-byte block of words
 * m[i] = (16 g + i) * 0x9E3779B9 (mod 2^32), i = 0..15, little-endian, with counter j,
 * block length 64 and flags KEYED_HASH.  Chain g's final CV goes to d_cvs + 32 g
 * (32 / lanes_per_chunk CVs, 16-byte aligned) and the clock cycles of lane 0's whole
 * chain to *d_cycles (8-byte aligned): the dependency-chain latency of one compression
 * is *d_cycles / chain.  Asynchronous.
 * Errors: B3G_ERR_NULL, B3G_ERR_ARG, B3G_ERR_ALIGN, B3G_ERR_CUDA.
 */
b3g_status blake3_selftest_compress_latency(int lanes_per_chunk, uint32_t chain, const uint8_t key[32],
                                            uint8_t *d_cvs, uint64_t *d_cycles, b3g_stream_t stream);

/*
 * blake3_selftest_compress_rate -- launches `blocks` CTAs of 128 threads (1..2^20) on
 * `stream`; every thread runs `iters` (1..2^20) chained keyed compressions with the
 * same compression function as the hashing kernels, its 16 message words held in
 * registers, and touches no memory but the 4-byte device word d_sink (written only on
 * an impossible value).  blocks * 128 * iters compressions per launch: the
 * compression-only ceiling, for the caller to time (asynchronous).  The compression
 * is the one the page describes in its section "压缩函数" (7 rounds of G).
 * Errors: B3G_ERR_NULL, B3G_ERR_ARG, B3G_ERR_ALIGN (d_sink not 4-byte aligned),
 * B3G_ERR_CUDA.
 */
b3g_status blake3_selftest_compress_rate(uint32_t blocks, uint32_t iters, uint32_t *d_sink,
                                         b3g_stream_t stream);

/*
 * blake3_keyed_hash_xof -- out_len bytes of extendable output for d_in[0..len) under
 * `key`, written to d_out (any alignment).  The first 32 bytes equal the digest of
 * blake3_keyed_hash.  Output block i (bytes 64i .. 64i+63) is the root compression
 * with ROOT set and its counter equal to i (BLAKE3 specification, extendable output;
 * the page lists this mode under "未来工作" as not implemented).  Temporary device
 * memory comes from the stream-ordered allocator.
 * Errors: B3G_ERR_NULL, B3G_ERR_ARG (out_len beyond 2^31 * 16 KiB), B3G_ERR_CUDA.
 */
b3g_status blake3_keyed_hash_xof(const void *d_in, uint64_t len, const uint8_t key[32],
                                 uint8_t *d_out, uint64_t out_len, b3g_stream_t stream);

/* blake3_hash_xof -- extendable output in the default (unkeyed) mode; otherwise as
 * blake3_keyed_hash_xof. */
b3g_status blake3_hash_xof(const void *d_in, uint64_t len, uint8_t *d_out, uint64_t out_len,
                           b3g_stream_t stream);

/*
 * Streaming hasher: the digest of input that arrives as successive device segments of
 * any length, equal to the digest of their concatenation.  The hasher is a host object
 * that owns, on the device current at creation, about 3 KiB of device memory, a side
 * stream of the highest priority and three events; the first update shorter than
 * 64 MiB that does not fit in what is buffered adds a 64 MiB accumulation buffer
 * (cudaMalloc; if that fails the hasher goes on without it).  Every call must be made
 * with that device current (else B3G_ERR_ARG).  Calls are asynchronous on the stream
 * passed; a hasher must be used from one stream at a time (calls in stream order), and
 * a segment may be reused once the update's work on that stream is done.  Segments
 * are copied into the accumulation buffer while they fit and pushed in large batches;
 * whole runs of chunks go through the same leaf and reduction kernels as
 * blake3_keyed_hash, and the small launches after them run on the side stream, joined
 * back to the caller's stream by events (fully, when the caller's stream is being
 * captured into a graph).  Chaining values are merged only once more input is known to
 * follow (page section "BLAKE3": the tree rules).
 */
typedef struct b3g_hasher b3g_hasher;

/* Creates a hasher for `key` (host pointer, copied).  Allocates with cudaMalloc and
 * creates its side stream and events. */
b3g_status blake3_hasher_new(const uint8_t key[32], b3g_hasher **out);

/* Creates a hasher in the default (unkeyed) mode (see blake3_hash); otherwise as
 * blake3_hasher_new. */
b3g_status blake3_hasher_new_default(b3g_hasher **out);

/* Frees the hasher, its device memory, stream and events (waits for its side stream;
 * cudaFree synchronises the device). */
void blake3_hasher_free(b3g_hasher *h);

/* Forgets all input (same key).  Host-side only. */
b3g_status blake3_hasher_reset(b3g_hasher *h);

/* Bytes absorbed so far. */
uint64_t blake3_hasher_count(const b3g_hasher *h);

/* Absorbs d_in[0..len).  Errors: B3G_ERR_NULL, B3G_ERR_ARG, B3G_ERR_CUDA.  After an
 * error the hasher's contents are unspecified: reset it before using it again. */
b3g_status blake3_hasher_update(b3g_hasher *h, const void *d_in, uint64_t len, b3g_stream_t stream);

/* Absorbs count device segments in order, d_ptrs[i][0..lens[i]) (host arrays of device
 * pointers and lengths), with the result of count blake3_hasher_update calls.  Runs of
 * segments that fit in the accumulation buffer are copied by one gather launch per up
 * to 1024 segments (128 when fewer are left), so many small segments cost one launch
 * instead of one copy each.
 * Errors: B3G_ERR_NULL (h NULL; d_ptrs or lens NULL with count > 0; a NULL pointer with
 * a nonzero length), B3G_ERR_ARG, B3G_ERR_CUDA. */
b3g_status blake3_hasher_update_many(b3g_hasher *h, const void *const *d_ptrs, const uint64_t *lens,
                                     uint64_t count, b3g_stream_t stream);

/*
 * Checkpoint and resume.  blake3_hasher_export writes the hasher's whole state (mode,
 * key, counts, the stack of subtree CVs and the bytes not yet pushed: at most about
 * 64 MiB, blake3_hasher_export_size bytes) to host memory h_buf, after the work queued
 * on `stream` (it synchronises the stream); the hasher is not changed.
 * blake3_hasher_import creates a hasher on the current device from such a record, so
 * that hashing can go on in another process or on another device with the same result.
 * The record is little-endian and starts with "B3GH" and a version number.
 * Errors: B3G_ERR_NULL; B3G_ERR_WORKSPACE (export buffer too small); B3G_ERR_ARG
 * (import of a record that is not a state the hasher can reach: checked before any
 * CUDA call); B3G_ERR_CUDA.
 */
size_t blake3_hasher_export_size(const b3g_hasher *h);
b3g_status blake3_hasher_export(const b3g_hasher *h, void *h_buf, size_t buf_bytes, b3g_stream_t stream);
b3g_status blake3_hasher_import(const void *h_buf, size_t buf_bytes, b3g_hasher **out, b3g_stream_t stream);

/* Writes out_len bytes of output (32 for the digest) to d_out.  The hasher is not
 * changed: more input may follow.  Errors: B3G_ERR_NULL, B3G_ERR_ARG, B3G_ERR_CUDA. */
b3g_status blake3_hasher_finalize(const b3g_hasher *h, uint8_t *d_out, uint64_t out_len,
                                  b3g_stream_t stream);

/*
 * blake3_keyed_hash_host -- the digest of HOST memory h_in[0..len), written to the host
 * buffer out32.  The input is copied to the device in segments on an internal copy
 * stream, into two alternating slots of the device buffer d_staging, while the other
 * slot is hashed on `stream` by the streaming hasher (copies and hashing overlap).
 * For full speed h_in should be page-locked (cudaHostAlloc / cudaHostRegister).
 * d_staging (256-byte aligned, at least 3328 + 2 MiB bytes; its size sets the segment
 * size) may be NULL: then 128 MiB + 3328 bytes come from the stream-ordered allocator.
 * Synchronous: returns once the digest is in out32.
 * Errors: B3G_ERR_NULL, B3G_ERR_ALIGN, B3G_ERR_WORKSPACE (d_staging too small),
 * B3G_ERR_CUDA.
 */
b3g_status blake3_keyed_hash_host(const void *h_in, uint64_t len, const uint8_t key[32],
                                  uint8_t out32[32], void *d_staging, size_t staging_bytes,
                                  b3g_stream_t stream);

/* blake3_hash_host -- the default-mode (unkeyed) digest of host memory; otherwise as
 * blake3_keyed_hash_host. */
b3g_status blake3_hash_host(const void *h_in, uint64_t len, uint8_t out32[32], void *d_staging,
                            size_t staging_bytes, b3g_stream_t stream);

/*
 * blake3_keyed_hash_noalloc -- the same digest as blake3_keyed_hash, computed without
 * allocating any device memory.  The page has no counterpart to this entry point.
 *
 * For callers that cannot allocate device memory when they hash: for example a
 * process whose GPU memory is already owned by another allocator (a framework's
 * caching allocator), a latency-critical loop that cannot accept the device-wide
 * synchronisation cudaMalloc/cudaFree may cause, or a service that forbids allocation
 * after start-up.  The CTA roots and the leaf kernel's tile counter are kept in a
 * fixed scratch array of 4 MiB + 8 KiB that is part of the library's device image:
 * every GPU that loads libb3g.so holds it until the process exits.  The caller still
 * provides the input and the 32-byte, 16-byte aligned output.  The kernels and CTA
 * subtree sizes are those of blake3_keyed_hash.
 *
 * Limits and rules:
 *   - len may be at most B3G_NOALLOC_MAX_LEN (16 GiB); a larger input returns
 *     B3G_ERR_WORKSPACE before anything is launched.
 *   - The first call on each device looks up the scratch array's device address
 *     (with that device current) and caches it; make that first call before any
 *     stream capture on that device.
 *   - All calls share the one scratch array, and it keeps the last call's contents.
 *     Calls whose work overlaps on the GPU (concurrent streams, or several host
 *     threads on one device) race on it and give wrong digests; serialise them.
 *     Within one call everything read from the scratch is written first (the tile
 *     counter is cleared by a one-thread kernel on `stream`), so leftovers of an
 *     earlier call do no harm.
 * Errors: B3G_ERR_NULL, B3G_ERR_ALIGN (d_out32), B3G_ERR_WORKSPACE (len too large),
 * B3G_ERR_CUDA.
 */
#define B3G_NOALLOC_MAX_LEN (16ull << 30)
b3g_status blake3_keyed_hash_noalloc(const void *d_in, uint64_t len, const uint8_t key[32],
                                     uint8_t *d_out32, b3g_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BLAKE3_GB300_H */

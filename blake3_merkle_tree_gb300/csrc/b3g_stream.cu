// b3g_stream.cu -- extendable output and the streaming (segmented) hasher.
//
// Source page: "BLAKE3 GPU 400x faster hashing" (qfminer.top).
//   section "未来工作": the extendable-output mode (XOF) is listed as not implemented.
//   section "BLAKE3": the tree rules (left subtree full, left subtree at least as
//     large), which decide when chaining values may be merged.
// The output mode follows the BLAKE3 specification (O'Connor et al., 2020, section
// 2.6): the root compression is kept as its inputs, and output block i (64 bytes) is
// that compression with ROOT set and the counter equal to i.
//
// Extendable output: the root's inputs ("root record": CV, message block, block
// length, flags) are produced on the device, then xof_kernel writes every output
// block in parallel, one thread per 64-byte block.
//   - one chunk: the record is the chunk's last block, the CV chained through the
//     blocks before it;
//   - several chunks: the record is the top parent, whose children are the largest
//     power-of-two left subtree and the rest; both are ordinary subtree roots.
//
// Streaming hasher: input arrives in device segments of any length.  A small device
// state holds a stack of subtree CVs; bytes not yet pushed wait in an accumulation
// buffer (1024 bytes inside the state, later an own 64 MiB buffer); the host tracks
// the counts.
//   - Segments are copied into the buffer while they fit.  When one does not, the
//     buffer's chunks are pushed, and so are the segment's whole chunks if they do not
//     fit in the buffer either; what is left is kept.  Nothing is pushed while the
//     input is at most one chunk (that chunk may turn out to be the whole input and
//     then needs ROOT).
//   - Whole runs of chunks are pushed as aligned power-of-two subtrees computed by
//     the ordinary leaf and reduction kernels; a subtree pushed at position 0 is
//     pushed as its two halves, so that the root's two children always exist.
//   - Before pushing at chunk position p the stack is merged down to popcount(p)
//     entries (the binary decomposition of p), so merges happen only once it is
//     known that more input follows.
//   - Finalize works on a copy of the stack: the buffered chunks but the last are
//     pushed onto it, the last (possibly partial) chunk is appended, the copy is
//     merged down to max(2, popcount(n)) entries and folded right to left; the bottom
//     entry and the fold are the root's children.  The hasher can keep absorbing
//     input afterwards.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "b3g_device.cuh"
#include "b3g_internal.h"

namespace b3g {
namespace {

constexpr int kStackSlots = 66;
// device state of a hasher: [stack 66 x 32 B][chunk buffer 1024 B][root record 128 B]
constexpr size_t kStackBytes = kStackSlots * 32;
constexpr size_t kBufOff = kStackBytes;
constexpr size_t kRecordOff = kBufOff + 1024;
constexpr size_t kStateBytes = kRecordOff + 128;
// root record words: cv[0..7], block[8..23], block_len[24], flags[25] (ROOT not set)
constexpr int kRecWords = 26;

// The `len` (0..1024) bytes at `p` as 256 little-endian words, zero past len, in
// `words`; every thread of the block takes a share of the byte loads (any alignment).
__device__ void stage_chunk(const uint8_t *p, uint32_t len, uint32_t *words) {
    for (uint32_t w = threadIdx.x; w < 256u; w += blockDim.x) {
        uint32_t v = 0;
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k) {
            const uint32_t i = 4u * w + k;
            if (i < len) v |= static_cast<uint32_t>(p[i]) << (8u * k);
        }
        words[w] = v;
    }
}

// Root record of one chunk of `len` (0..1024) bytes, staged by stage_chunk, with
// counter ctr: the inputs of its last compression.
__device__ void chunk_record(const uint32_t *words, uint32_t len, uint64_t ctr, const uint32_t key[8],
                             uint32_t mode_flags, uint32_t *rec) {
    const uint32_t nblocks = len == 0 ? 1u : (len + 63u) / 64u;
    uint32_t cv[8];
    for (int i = 0; i < 8; ++i) cv[i] = key[i];
    uint32_t m[16];
    for (uint32_t b = 0; b + 1 < nblocks; ++b) {
        for (int i = 0; i < 16; ++i) m[i] = words[16 * b + i];
        compress(cv, m, static_cast<uint32_t>(ctr), static_cast<uint32_t>(ctr >> 32), 64u,
                 mode_flags | (b == 0 ? kChunkStart : 0u));
    }
    const uint32_t b = nblocks - 1;
    for (int i = 0; i < 8; ++i) rec[i] = cv[i];
    for (int i = 0; i < 16; ++i) rec[8 + i] = words[16 * b + i];
    rec[24] = len - 64u * b;
    rec[25] = mode_flags | kChunkEnd | (b == 0 ? kChunkStart : 0u);
}

// CV (no ROOT) of one chunk staged by stage_chunk.
__device__ void chunk_cv(const uint32_t *words, uint32_t len, uint64_t ctr, const uint32_t key[8],
                         uint32_t mode_flags, uint32_t cv[8]) {
    uint32_t r[kRecWords];
    chunk_record(words, len, ctr, key, mode_flags, r);
    uint32_t m[16];
    for (int i = 0; i < 8; ++i) cv[i] = r[i];
    for (int i = 0; i < 16; ++i) m[i] = r[8 + i];
    compress(cv, m, static_cast<uint32_t>(ctr), static_cast<uint32_t>(ctr >> 32), r[24], r[25]);
}

// Merge the top of a stack of CVs (8 words each) down to `target` entries.
__device__ uint32_t merge_down(uint32_t *st, uint32_t depth, uint32_t target, const uint32_t key[8],
                               uint32_t mode_flags) {
    while (depth > target) {
        uint32_t l[8], r[8], p[8];
        for (int i = 0; i < 8; ++i) {
            l[i] = st[8 * (depth - 2) + i];
            r[i] = st[8 * (depth - 1) + i];
        }
        parent(key, mode_flags, l, r, false, p);
        for (int i = 0; i < 8; ++i) st[8 * (depth - 2) + i] = p[i];
        --depth;
    }
    return depth;
}

enum RecordMode : uint32_t {
    kRecChunk = 0,     // root record of the single chunk at `in`
    kRecPush = 1,      // merge the stack to `target`, push the CV of the full chunk at `in`
    kRecFinalize = 2,  // root record of the whole input, last chunk at `in` (stack untouched)
    kRecMerge = 3,     // merge the stack to `target`
    kRecParent = 4,    // record = (key, message words already in place, 64, KEYED_HASH|PARENT)
    kRecPushMany = 5,  // for each piece in order: merge to popcount(position), push its root
};

constexpr int kMaxPieces = 96;        // pieces of one update on the batched path
constexpr int kMaxSmallPieces = 16;   // pieces shorter than one CTA subtree (head and tail)

struct RecordArgs {
    const uint8_t *in;  // the chunk bytes (kRecChunk, kRecPush, kRecFinalize)
    uint8_t *state;     // hasher state, or a scratch area laid out the same way
    uint64_t pushed;    // chunks whose CVs are in the stack (= counter of the next chunk)
    uint32_t len;       // bytes of the chunk to finish (kRecChunk, kRecPush, kRecFinalize)
    uint32_t depth;     // stack entries
    uint32_t target;    // stack entries after merging (kRecPush, kRecMerge)
    uint32_t mode;
    uint32_t key[8];      // the key, or the IV in the default mode
    uint32_t mode_flags;  // flag bits of the hash mode on every compression
    // kRecPushMany: roots of `npieces` pieces (32 bytes each) and their chunk positions
    const uint8_t *roots;
    uint32_t npieces;
    uint64_t piece_pos[kMaxPieces];
};

// The sequential bookkeeping of the hasher: at most 65 merges and one chunk per
// launch, a chain of dependent compressions that lane 0 runs alone.  The warp first
// stages everything the chain reads (the CV stack, the piece roots, the chunk bytes)
// in shared memory, so that the chain pays one round of global loads instead of one
// per step, and afterwards writes the stack back.
__global__ void __launch_bounds__(32) record_kernel(const RecordArgs a) {
    __shared__ uint32_t s_stack[kStackSlots * 8];
    __shared__ uint32_t s_roots[kMaxPieces * 8];
    __shared__ uint32_t s_chunk[256];
    __shared__ uint32_t s_depth;
    const uint32_t lane = threadIdx.x;
    uint32_t *stack = reinterpret_cast<uint32_t *>(a.state);
    uint32_t *rec = reinterpret_cast<uint32_t *>(a.state + kRecordOff);
    const bool reads_stack = a.mode == kRecMerge || a.mode == kRecPush || a.mode == kRecPushMany ||
                             a.mode == kRecFinalize;
    if (reads_stack)
        for (uint32_t i = lane; i < 8u * a.depth; i += 32u) s_stack[i] = stack[i];
    if (a.mode == kRecPushMany) {
        const uint32_t *rw = reinterpret_cast<const uint32_t *>(a.roots);
        for (uint32_t i = lane; i < 8u * a.npieces; i += 32u) s_roots[i] = rw[i];
    }
    if (a.mode == kRecChunk || (a.mode == kRecFinalize && a.len > 0)) stage_chunk(a.in, a.len, s_chunk);
    if (a.mode == kRecPush) stage_chunk(a.in, 1024u, s_chunk);
    __syncwarp();

    if (lane == 0) {
        uint32_t key[8];
        for (int i = 0; i < 8; ++i) key[i] = a.key[i];
        uint32_t keep = 0;  // stack entries to write back
        switch (a.mode) {
            case kRecChunk:
                chunk_record(s_chunk, a.len, a.pushed, key, a.mode_flags, rec);
                break;
            case kRecMerge:
                keep = merge_down(s_stack, a.depth, a.target, key, a.mode_flags);
                break;
            case kRecPush: {
                const uint32_t d = merge_down(s_stack, a.depth, a.target, key, a.mode_flags);
                chunk_cv(s_chunk, 1024u, a.pushed, key, a.mode_flags, s_stack + 8 * d);
                keep = d + 1;
                break;
            }
            case kRecPushMany: {
                uint32_t d = a.depth;
                for (uint32_t j = 0; j < a.npieces; ++j) {
                    d = merge_down(s_stack, d, static_cast<uint32_t>(__popcll(a.piece_pos[j])), key, a.mode_flags);
                    for (int i = 0; i < 8; ++i) s_stack[8 * d + i] = s_roots[8 * j + i];
                    ++d;
                }
                keep = d;
                break;
            }
            case kRecParent:
                for (int i = 0; i < 8; ++i) rec[i] = key[i];
                rec[24] = kBlockLen;
                rec[25] = a.mode_flags | kParent;
                break;
            case kRecFinalize: {
                // the staged stack is a private copy: the hasher state is not changed
                uint32_t *st = s_stack;
                uint32_t d = a.depth;
                uint64_t n = a.pushed;
                if (a.len > 0) {  // the unfinished chunk becomes the last leaf
                    d = merge_down(st, d, static_cast<uint32_t>(__popcll(n)), key, a.mode_flags);
                    chunk_cv(s_chunk, a.len, n, key, a.mode_flags, st + 8 * d);
                    ++d;
                    ++n;
                }
                const uint32_t pc = static_cast<uint32_t>(__popcll(n));
                d = merge_down(st, d, pc < 2 ? 2u : pc, key, a.mode_flags);
                uint32_t cv[8];
                for (int i = 0; i < 8; ++i) cv[i] = st[8 * (d - 1) + i];
                for (uint32_t e = d - 1; e > 1; --e) {
                    uint32_t l[8];
                    for (int i = 0; i < 8; ++i) l[i] = st[8 * (e - 1) + i];
                    parent(key, a.mode_flags, l, cv, false, cv);
                }
                for (int i = 0; i < 8; ++i) {
                    rec[i] = key[i];
                    rec[8 + i] = st[i];
                    rec[16 + i] = cv[i];
                }
                rec[24] = kBlockLen;
                rec[25] = a.mode_flags | kParent;
                break;
            }
            default:
                break;
        }
        s_depth = keep;
    }
    __syncwarp();
    const uint32_t keep = s_depth;
    for (uint32_t i = lane; i < 8u * keep; i += 32u) stack[i] = s_stack[i];
}

// Small pieces (at most 64 full chunks each, counters from `counter`), one CTA per
// piece, plain loads (any alignment): root of each piece (a perfect subtree, no ROOT).
struct PiecesArgs {
    const uint8_t *base;  // piece j starts at base + off[j]
    uint8_t *out;         // root of piece j at out + 32 * slot[j]
    uint32_t key[8];
    uint32_t mode_flags;
    uint64_t off[kMaxSmallPieces];
    uint64_t counter[kMaxSmallPieces];
    uint32_t nchunks[kMaxSmallPieces];
    uint32_t slot[kMaxSmallPieces];
};

__global__ void __launch_bounds__(64) pieces_kernel(const PiecesArgs a) {
    __shared__ __align__(128) uint8_t node_mem[64 * 32];
    const uint32_t nodes = smem_u32(node_mem);
    const uint32_t j = blockIdx.x, r = threadIdx.x;
    const uint32_t cnt = a.nchunks[j];
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = a.key[i];
    if (r < cnt) {
        const uint8_t *p = a.base + a.off[j] + 1024ull * r;
        const uint64_t ctr = a.counter[j] + r;
        uint32_t cv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[i] = key[i];
#pragma unroll 1
        for (uint32_t b = 0; b < 16; ++b) {
            uint32_t m[16];
            load_block_global(p, 1024, 64ull * b, m);
            const uint32_t flags = a.mode_flags | (b == 0 ? kChunkStart : 0u) | (b == 15 ? kChunkEnd : 0u);
            compress(cv, m, static_cast<uint32_t>(ctr), static_cast<uint32_t>(ctr >> 32), 64u, flags);
        }
        store_node(nodes, r, cv);
    }
    named_bar_sync(1, 64);
    uint32_t root[8];
    block_tree(nodes, cnt, r, 64, 1, key, a.mode_flags, false, root);
    if (r == 0) {
        uint4 *o = reinterpret_cast<uint4 *>(a.out + 32ull * a.slot[j]);
        o[0] = make_uint4(root[0], root[1], root[2], root[3]);
        o[1] = make_uint4(root[4], root[5], root[6], root[7]);
    }
}

// Each CTA reduces one range of `count` CVs (a power of two, at most 1024: a perfect
// subtree) starting at in + 32 * start, to out + 32 * slot (no ROOT).
struct RangesArgs {
    const uint8_t *in;
    uint8_t *out;
    uint32_t key[8];
    uint32_t mode_flags;
    uint32_t start[kMaxPieces];
    uint32_t count[kMaxPieces];
    uint32_t slot[kMaxPieces];
};

__global__ void __launch_bounds__(512) ranges_reduce_kernel(const RangesArgs a) {
    __shared__ __align__(128) uint8_t node_mem[512 * 32];
    const uint32_t nodes = smem_u32(node_mem);
    const uint32_t j = blockIdx.x, tid = threadIdx.x;
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = a.key[i];
    const uint32_t m = a.count[j];
    const uint8_t *in = a.in + 32ull * a.start[j];
    const uint32_t half = m >> 1;
    if (tid < half) {
        const uint4 *p = reinterpret_cast<const uint4 *>(in + 64ull * tid);
        const uint4 w0 = p[0], w1 = p[1], w2 = p[2], w3 = p[3];
        uint32_t l[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t r[8] = {w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
        uint32_t res[8];
        parent(key, a.mode_flags, l, r, false, res);
        store_node(nodes, tid, res);
    } else if (m == 1 && tid == 0) {
        const uint4 *p = reinterpret_cast<const uint4 *>(in);
        const uint4 w0 = p[0], w1 = p[1];
        uint32_t res[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        store_node(nodes, 0, res);
    }
    named_bar_sync(1, blockDim.x);
    uint32_t root[8];
    block_tree(nodes, m == 1 ? 1u : half, tid, blockDim.x, 1, key, a.mode_flags, false, root);
    if (tid == 0) {
        uint4 *o = reinterpret_cast<uint4 *>(a.out + 32ull * a.slot[j]);
        o[0] = make_uint4(root[0], root[1], root[2], root[3]);
        o[1] = make_uint4(root[4], root[5], root[6], root[7]);
    }
}

// Gather copy for blake3_hasher_update_many: segment j (src[j], len[j] bytes) goes to
// dst + off[j]; the copy is cut into pieces of kGatherPiece bytes, piece0[j] being
// segment j's first piece, and CTA i copies piece i.  A piece whose source and
// destination share their alignment modulo 16 moves 16-byte words between a byte head
// and a byte tail; any other piece moves bytes.  The segment table travels in the
// kernel parameters: K = 128 entries (3.6 KB) for short calls, K = 1024 (28 KB, under
// the 32,764-byte parameter limit) when more segments are waiting, so that a call with
// many small segments needs an eighth of the launches.
constexpr int kGatherSmall = 128;
constexpr int kGatherBig = 1024;
constexpr uint32_t kGatherPiece = 32 * 1024;

template <int K>
struct GatherArgs {
    uint8_t *dst;
    uint32_t n;
    const uint8_t *src[K];
    uint64_t off[K];
    uint64_t len[K];
    uint32_t piece0[K + 1];
};
static_assert(sizeof(GatherArgs<kGatherBig>) <= 32764, "kernel parameter limit");

template <int K>
__global__ void __launch_bounds__(256) gather_kernel(const GatherArgs<K> a) {
    const uint32_t piece = blockIdx.x;
    uint32_t lo = 0, hi = a.n;  // the segment j with piece0[j] <= piece < piece0[j + 1]
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) / 2;
        if (a.piece0[mid] <= piece) lo = mid;
        else hi = mid;
    }
    const uint32_t j = lo;
    const uint64_t p0 = static_cast<uint64_t>(piece - a.piece0[j]) * kGatherPiece;
    const uint64_t p1 = a.len[j] - p0 < kGatherPiece ? a.len[j] : p0 + kGatherPiece;
    const uint8_t *src = a.src[j];
    uint8_t *dst = a.dst + a.off[j];
    const uint32_t t = threadIdx.x, nt = blockDim.x;
    const uintptr_t sa = reinterpret_cast<uintptr_t>(src + p0), da = reinterpret_cast<uintptr_t>(dst + p0);
    if ((sa & 15u) == (da & 15u)) {
        uint64_t head = (16u - (sa & 15u)) & 15u;
        head = head < p1 - p0 ? head : p1 - p0;
        for (uint64_t i = t; i < head; i += nt) dst[p0 + i] = src[p0 + i];
        const uint64_t q0 = p0 + head;
        const uint64_t nvec = (p1 - q0) / 16;
        const uint4 *sv = reinterpret_cast<const uint4 *>(src + q0);
        uint4 *dv = reinterpret_cast<uint4 *>(dst + q0);
        for (uint64_t i = t; i < nvec; i += nt) dv[i] = sv[i];
        for (uint64_t i = q0 + 16 * nvec + t; i < p1; i += nt) dst[i] = src[i];
    } else {
        for (uint64_t i = p0 + t; i < p1; i += nt) dst[i] = src[i];
    }
}

struct XofArgs {
    const uint32_t *rec;  // root record (device)
    uint8_t *out;
    uint64_t out_len;
};

// Output block i = the root compression with counter i and ROOT, 64 bytes.
__global__ void __launch_bounds__(256) xof_kernel(const XofArgs a) {
    const uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i * 64 >= a.out_len) return;
    uint32_t cv[8], m[16], o[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) cv[k] = __ldg(a.rec + k);
#pragma unroll
    for (int k = 0; k < 16; ++k) m[k] = __ldg(a.rec + 8 + k);
    const uint32_t blen = __ldg(a.rec + 24);
    const uint32_t flags = __ldg(a.rec + 25) | kRoot;
    compress_full(cv, m, static_cast<uint32_t>(i), static_cast<uint32_t>(i >> 32), blen, flags, o);
    uint8_t *dst = a.out + i * 64;
    const uint64_t rest = a.out_len - i * 64;
    if (rest >= 64 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q) d4[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        return;
    }
    const uint32_t take = rest < 64 ? static_cast<uint32_t>(rest) : 64u;
#pragma unroll
    for (uint32_t k = 0; k < 64; ++k)
        if (k < take) dst[k] = static_cast<uint8_t>(o[k >> 2] >> (8 * (k & 3)));
}

b3g_status launch_record(const RecordArgs &a, cudaStream_t s) {
    record_kernel<<<1, 32, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "record_kernel launch");
}

b3g_status launch_xof(const uint32_t *rec, uint8_t *out, uint64_t out_len, cudaStream_t s) {
    if (out_len == 0) return B3G_OK;
    const uint64_t blocks = (out_len + 63) / 64;
    const uint64_t grid = (blocks + 255) / 256;
    if (grid > 0x7fffffffull) return B3G_ERR_ARG;
    XofArgs xa{rec, out, out_len};
    xof_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(xa);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "xof_kernel launch");
}

uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

uint32_t popcount64(uint64_t x) { return static_cast<uint32_t>(__builtin_popcountll(x)); }

void key_words(const uint8_t key[32], uint32_t out[8]) {
    for (int i = 0; i < 8; ++i)
        out[i] = static_cast<uint32_t>(key[4 * i]) | (static_cast<uint32_t>(key[4 * i + 1]) << 8) |
                 (static_cast<uint32_t>(key[4 * i + 2]) << 16) | (static_cast<uint32_t>(key[4 * i + 3]) << 24);
}

RecordArgs record_args(uint8_t *state, const uint32_t key[8], uint32_t mode_flags, uint32_t mode) {
    RecordArgs ra;
    std::memset(&ra, 0, sizeof ra);
    ra.state = state;
    std::memcpy(ra.key, key, sizeof ra.key);
    ra.mode_flags = mode_flags;
    ra.mode = mode;
    return ra;
}

b3g_status check_device(int want) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    return dev == want ? B3G_OK : B3G_ERR_ARG;
}

// Per-device streams kept for the life of the process, created on first use: kind 0
// carries the staging copies of blake3_keyed_hash_host, kind 1 is the side stream of
// its hasher (created with the highest priority, like a hasher's own side stream).
b3g_status cached_stream(int kind, cudaStream_t *out) {
    static std::mutex mu;
    static cudaStream_t cache[2][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64 || kind < 0 || kind > 1) return B3G_ERR_ARG;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[kind][dev]) {
        int least = 0, greatest = 0;
        e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess)
            e = cudaStreamCreateWithPriority(&cache[kind][dev], cudaStreamNonBlocking, kind == 1 ? greatest : least);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithPriority");
    }
    *out = cache[kind][dev];
    return B3G_OK;
}

}  // namespace
}  // namespace b3g

using namespace b3g;

// Host object of a streaming hasher (opaque to callers).
//
// Bytes absorbed but not yet pushed live in `acc`: at first the 1024-byte buffer inside
// the state, then (on the first update that would otherwise start a push for a segment
// shorter than kAccBytes) an own kAccBytes buffer, so that a stream of small segments
// costs one device copy each and the chunks are pushed in large batches.  Work that
// needs no SM-wide parallelism (small pieces, range reductions, the sequential stack
// records) runs on the high-priority side stream `aux`, ordered against the caller's
// stream with events, so that it overlaps the leaf launches on the caller's stream.
//
// A hasher of its own (blake3_hasher_new) has a second side stream, `rd`, for the work
// that reads the caller's segment or acc: the small pieces and the copy of a single
// pushed chunk into one of kChunkSlots staging slots.  The caller's stream then waits
// only for those reads before it reuses the segment or rewrites acc, not for the chain
// of records and reductions queued on `aux`, which waits for every leaf launch and runs
// slowly while the next leaf launch fills the SMs.
constexpr int kChunkSlots = 4;

struct b3g_hasher {
    uint8_t key[32];      // the key, or the IV (little-endian) in the default mode
    uint32_t kw[8];
    uint32_t mode_flags;  // KEYED_HASH in keyed mode, none in the default mode
    uint8_t *state;     // device: stack, 1024-byte chunk buffer, root record
    uint8_t *acc;       // device: bytes absorbed but not pushed (the state's buffer or own)
    uint64_t acc_cap;   // capacity of acc: 1024, or kAccBytes once grown
    uint64_t acc_len;   // bytes in acc
    bool may_grow;      // may switch acc to an own kAccBytes buffer
    bool own_streams;   // aux and the events belong to this object
    bool read_pending;  // aux has reads of a segment or of acc that the caller's stream has not waited for
    int device;
    uint64_t count;     // bytes absorbed
    uint64_t pushed;    // chunks whose CVs are represented in the stack
    uint32_t depth;     // stack entries
    cudaStream_t aux;   // side stream
    cudaEvent_t ev_fork, ev_read, ev_done;
    cudaStream_t rd;    // second side stream (NULL: everything on aux)
    cudaEvent_t ev_fork_rd, ev_read_rd, ev_rd_done, ev_rd_all;
    bool rd_pending;    // rd has reads that the caller's stream has not waited for
    uint8_t *slots;     // device: kChunkSlots staging slots of 1024 bytes (with rd)
    cudaEvent_t ev_slot[kChunkSlots];  // recorded on aux after the chain read slot k
    uint32_t slot_next;
};

namespace {

constexpr uint64_t kAccBytes = 64ull << 20;

// aux waits until `s` reaches this point
b3g_status fork_aux(b3g_hasher *h, cudaStream_t s) {
    cudaError_t e = cudaEventRecord(h->ev_fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->aux, h->ev_fork, 0);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "fork to the side stream");
}

// the side stream's reads of segments and of acc, so far, end here
b3g_status mark_read(b3g_hasher *h) {
    cudaError_t e = cudaEventRecord(h->ev_read, h->aux);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    h->read_pending = true;
    return B3G_OK;
}

// rd waits until `s` reaches this point
b3g_status fork_rd(b3g_hasher *h, cudaStream_t s) {
    cudaError_t e = cudaEventRecord(h->ev_fork_rd, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->rd, h->ev_fork_rd, 0);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "fork to the readers' stream");
}

// rd's reads of segments and of acc, so far, end here; and aux waits for rd's work so
// far (the piece roots, a staged chunk) before its next launch
b3g_status rd_handoff(b3g_hasher *h) {
    cudaError_t e = cudaEventRecord(h->ev_read_rd, h->rd);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_rd_done, h->rd);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->aux, h->ev_rd_done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "hand over from the readers' stream");
    h->rd_pending = true;
    return B3G_OK;
}

// `s` waits for those reads: afterwards the segment may be reused and acc rewritten
b3g_status join_reads(b3g_hasher *h, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (h->read_pending) e = cudaStreamWaitEvent(s, h->ev_read, 0);
    if (e == cudaSuccess && h->rd_pending) e = cudaStreamWaitEvent(s, h->ev_read_rd, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
    h->read_pending = h->rd_pending = false;
    return B3G_OK;
}

// `s` waits for everything queued on the side streams
b3g_status join_all(b3g_hasher *h, cudaStream_t s) {
    cudaError_t e = cudaEventRecord(h->ev_done, h->aux);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_done, 0);
    if (e == cudaSuccess && h->rd) e = cudaEventRecord(h->ev_rd_all, h->rd);
    if (e == cudaSuccess && h->rd) e = cudaStreamWaitEvent(s, h->ev_rd_all, 0);
    if (e != cudaSuccess) return cuda_fail(e, "join the side stream");
    h->read_pending = h->rd_pending = false;
    return B3G_OK;
}

b3g_status streams_init(b3g_hasher *h, bool own) {
    h->own_streams = own;
    h->read_pending = h->rd_pending = false;
    h->aux = h->rd = nullptr;
    h->ev_fork = h->ev_read = h->ev_done = nullptr;
    h->ev_fork_rd = h->ev_read_rd = h->ev_rd_done = h->ev_rd_all = nullptr;
    h->slots = nullptr;
    for (cudaEvent_t &ev : h->ev_slot) ev = nullptr;
    h->slot_next = 0;
    cudaError_t e = cudaSuccess;
    if (own) {
        int least = 0, greatest = 0;
        e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->aux, cudaStreamNonBlocking, greatest);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithPriority");
    } else {
        b3g_status st = cached_stream(1, &h->aux);
        if (st != B3G_OK) return st;
    }
    cudaEvent_t *evs[3] = {&h->ev_fork, &h->ev_read, &h->ev_done};
    for (cudaEvent_t *ev : evs)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreateWithFlags");
    if (!own) return B3G_OK;
    // the readers' stream, its events and the chunk staging slots
    int least = 0, greatest = 0;
    e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->rd, cudaStreamNonBlocking, greatest);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithPriority");
    cudaEvent_t *rd_evs[4] = {&h->ev_fork_rd, &h->ev_read_rd, &h->ev_rd_done, &h->ev_rd_all};
    for (cudaEvent_t *ev : rd_evs)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (cudaEvent_t &ev : h->ev_slot)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreateWithFlags");
    e = alloc_sync(reinterpret_cast<void **>(&h->slots), kChunkSlots * kChunkBytes);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "chunk staging slots");
}

void streams_release(b3g_hasher *h) {
    if (h->aux) cudaStreamSynchronize(h->aux);
    if (h->rd) cudaStreamSynchronize(h->rd);
    cudaEvent_t evs[7] = {h->ev_fork, h->ev_read, h->ev_done, h->ev_fork_rd, h->ev_read_rd, h->ev_rd_done,
                          h->ev_rd_all};
    for (cudaEvent_t ev : evs)
        if (ev) cudaEventDestroy(ev);
    for (cudaEvent_t &ev : h->ev_slot) {
        if (ev) cudaEventDestroy(ev);
        ev = nullptr;
    }
    if (h->own_streams && h->aux) cudaStreamDestroy(h->aux);
    if (h->rd) cudaStreamDestroy(h->rd);  // only a hasher's own streams have rd
    if (h->slots) cudaFree(h->slots);
    h->aux = h->rd = nullptr;
    h->slots = nullptr;
    h->ev_fork = h->ev_read = h->ev_done = nullptr;
    h->ev_fork_rd = h->ev_read_rd = h->ev_rd_done = h->ev_rd_all = nullptr;
}

// The aligned power-of-two pieces of the chunk run [pos, pos + n): at every position
// the largest power of two that divides the position and fits; a piece that starts at
// chunk 0 is split into its two halves, so that the root's children stay separate.
struct Piece {
    uint64_t pos, size;
};

std::vector<Piece> decompose(uint64_t pos, uint64_t n) {
    std::vector<Piece> pieces;
    while (n > 0) {
        uint64_t size = 1;
        while (size * 2 <= n && (pos == 0 || (pos % (size * 2)) == 0)) size *= 2;
        if (pos == 0 && size >= 2) {
            pieces.push_back({0, size / 2});
            pieces.push_back({size / 2, size / 2});
        } else {
            pieces.push_back({pos, size});
        }
        pos += size;
        n -= size;
    }
    return pieces;
}

// One piece at a time, all on the side stream: a subtree launch per piece and a merge
// launch before each push.
b3g_status push_pieces_one_by_one(b3g_hasher *h, const uint8_t *p, const std::vector<Piece> &pieces,
                                  cudaStream_t s) {
    b3g_status st = fork_aux(h, s);
    if (st != B3G_OK) return st;
    const cudaStream_t x = h->aux;
    uint64_t biggest = 0;
    for (const Piece &pc : pieces) biggest = pc.size > biggest ? pc.size : biggest;
    const size_t ws_bytes = blake3_workspace_size(biggest * kChunkBytes);
    uint8_t *ws = nullptr;
    if (ws_bytes) {
        cudaError_t e = alloc_async(reinterpret_cast<void **>(&ws), ws_bytes, x);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync");
    }
    const uint64_t base = h->pushed;
    for (const Piece &pc : pieces) {
        const uint32_t target = popcount64(pc.pos);
        if (h->depth > target) {
            RecordArgs ra = record_args(h->state, h->kw, h->mode_flags, kRecMerge);
            ra.depth = h->depth;
            ra.target = target;
            st = launch_record(ra, x);
            if (st != B3G_OK) break;
            h->depth = target;
        }
        if (h->depth >= kStackSlots) {
            st = B3G_ERR_ARG;
            break;
        }
        st = hash_range_ws(p + (pc.pos - base) * kChunkBytes, pc.size * kChunkBytes, pc.pos, h->key, h->mode_flags, false,
                           h->state + 32ull * h->depth, ws, x);
        if (st != B3G_OK) break;
        h->depth += 1;
        h->pushed = pc.pos + pc.size;
    }
    if (ws) {
        cudaError_t e = cudaFreeAsync(ws, x);
        if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "cudaFreeAsync");
    }
    const b3g_status rs = mark_read(h);
    return st != B3G_OK ? st : rs;
}

// The record that merges the stack down and pushes the CV of the chunk at `src` (on the
// side stream); `slot` >= 0: `src` is that staging slot, released when the record has
// read it.
b3g_status push_record(b3g_hasher *h, const uint8_t *src, int slot) {
    RecordArgs ra = record_args(h->state, h->kw, h->mode_flags, kRecPush);
    ra.in = src;
    ra.depth = h->depth;
    ra.target = popcount64(h->pushed);
    ra.pushed = h->pushed;
    b3g_status st = launch_record(ra, h->aux);
    if (st == B3G_OK && slot >= 0) {
        const cudaError_t e = cudaEventRecord(h->ev_slot[slot], h->aux);
        if (e != cudaSuccess) st = cuda_fail(e, "cudaEventRecord");
    } else if (st == B3G_OK) {
        st = mark_read(h);
    }
    if (st == B3G_OK) {
        h->depth = ra.target + 1;
        h->pushed += 1;
    }
    return st;
}

// A staging slot for a chunk assembled on the readers' stream from up to two pieces
// (a, na bytes; then b, nb bytes; na + nb = 1024), after `s` has reached this point and
// the chain has released the slot.  Returns the slot's index in *slot.
b3g_status stage_chunk_rd(b3g_hasher *h, const uint8_t *a, uint64_t na, const uint8_t *b, uint64_t nb,
                          cudaStream_t s, int *slot) {
    const uint32_t k = h->slot_next++ % kChunkSlots;
    uint8_t *dst = h->slots + kChunkBytes * k;
    b3g_status st = fork_rd(h, s);
    if (st != B3G_OK) return st;
    cudaError_t e = cudaStreamWaitEvent(h->rd, h->ev_slot[k], 0);
    if (e == cudaSuccess && na) e = cudaMemcpyAsync(dst, a, na, cudaMemcpyDeviceToDevice, h->rd);
    if (e == cudaSuccess && nb) e = cudaMemcpyAsync(dst + na, b, nb, cudaMemcpyDeviceToDevice, h->rd);
    if (e != cudaSuccess) return cuda_fail(e, "chunk staging copy");
    *slot = static_cast<int>(k);
    return rd_handoff(h);
}

// One full chunk at `p`: a record launch on the side stream merges and pushes its CV.
// With the readers' stream the chunk is first copied there into a staging slot, which
// the record reads instead of `p`; under stream capture (the slots' events were
// recorded outside the capture) it is read in place.
b3g_status push_one(b3g_hasher *h, const uint8_t *p, cudaStream_t s) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const cudaError_t ce = cudaStreamIsCapturing(s, &cap);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamIsCapturing");
    if (h->rd && cap == cudaStreamCaptureStatusNone) {
        int slot = -1;
        const b3g_status st = stage_chunk_rd(h, p, kChunkBytes, nullptr, 0, s, &slot);
        return st == B3G_OK ? push_record(h, h->slots + kChunkBytes * slot, slot) : st;
    }
    const b3g_status st = fork_aux(h, s);
    return st == B3G_OK ? push_record(h, p, -1) : st;
}

// Push the chunks [h->pushed, h->pushed + nchunks) that start at `p`.  Batched: the
// pieces shorter than a CTA subtree (only at the two ends of the run) go through one
// launch of pieces_kernel on the side stream; the longer pieces are contiguous and
// aligned to a CTA subtree, so one leaf launch over their union (on `s`) yields their
// tile CVs, and one launch of ranges_reduce_kernel (plus the ordinary reduction for
// pieces of more than 1024 tiles) turns those into piece roots; one record_kernel
// launch then does every merge and push in order.  Everything after the leaf launch
// runs on the side stream.
b3g_status push_run(b3g_hasher *h, const uint8_t *p, uint64_t nchunks, cudaStream_t s) {
    if (nchunks == 1) return push_one(h, p, s);
    const std::vector<Piece> pieces = decompose(h->pushed, nchunks);
    const uint64_t tile = 1ull << kDefaultLeavesLog2;
    const uint64_t base = h->pushed;
    std::vector<size_t> small, big;
    for (size_t j = 0; j < pieces.size(); ++j) (pieces[j].size < tile ? small : big).push_back(j);
    uint64_t A = 0, B = 0;
    if (!big.empty()) {
        A = pieces[big.front()].pos;
        B = pieces[big.back()].pos + pieces[big.back()].size;
    }
    uint64_t big_sum = 0;
    for (size_t j : big) big_sum += pieces[j].size;
    if (stream_unbatched() || pieces.size() > static_cast<size_t>(kMaxPieces) ||
        small.size() > static_cast<size_t>(kMaxSmallPieces) ||
        big_sum != B - A || h->depth + pieces.size() >= static_cast<size_t>(kStackSlots) ||
        (B - A) / tile > 0xffffffffull)
        return push_pieces_one_by_one(h, p, pieces, s);

    // scratch: piece roots, tile CVs of [A, B), workspace of the large-piece reductions
    const uint64_t tiles = (B - A) / tile;
    size_t huge_ws = 0;
    for (size_t j : big) {
        const uint64_t t = pieces[j].size / tile;
        if (t > 1024) {
            const size_t w = blake3_reduce_workspace_size(t, -1);  // the group reduce_cvs_ws takes
            huge_ws = w > huge_ws ? w : huge_ws;
        }
    }
    const size_t roots_bytes = (pieces.size() * 32 + 255) & ~size_t(255);
    const size_t tiles_bytes = (tiles * 32 + 255) & ~size_t(255);
    uint8_t *scratch = nullptr;
    cudaError_t e = alloc_async(reinterpret_cast<void **>(&scratch), roots_bytes + tiles_bytes + huge_ws + 256, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync");
    uint8_t *roots = scratch;
    uint8_t *tile_cvs = scratch + roots_bytes;
    uint8_t *huge = tile_cvs + tiles_bytes;
    const cudaStream_t x = h->aux;
    // the side stream sees the segment and the scratch; so does the readers' stream,
    // which runs the small pieces when the hasher has one
    const cudaStream_t xp = h->rd && !small.empty() ? h->rd : x;
    b3g_status st = xp == x ? fork_aux(h, s) : fork_rd(h, s);
    if (st != B3G_OK) {
        cudaFreeAsync(scratch, s);
        return st;
    }

    if (!small.empty()) {
        PiecesArgs pa;
        std::memset(&pa, 0, sizeof pa);
        pa.base = p;
        pa.out = roots;
        std::memcpy(pa.key, h->kw, sizeof pa.key);
        pa.mode_flags = h->mode_flags;
        for (size_t i = 0; i < small.size(); ++i) {
            const Piece &pc = pieces[small[i]];
            pa.off[i] = (pc.pos - base) * kChunkBytes;
            pa.counter[i] = pc.pos;
            pa.nchunks[i] = static_cast<uint32_t>(pc.size);
            pa.slot[i] = static_cast<uint32_t>(small[i]);
        }
        pieces_kernel<<<static_cast<unsigned>(small.size()), 64, 0, xp>>>(pa);
        e = cudaGetLastError();
        // the roots go to the chain on aux (rd_handoff makes it wait for them)
        if (e != cudaSuccess) st = cuda_fail(e, "pieces_kernel launch");
        else st = xp == x ? mark_read(h) : rd_handoff(h);
    }
    if (st == B3G_OK && !big.empty()) {
        uint32_t *status = nullptr;
        st = device_status_word(&status);
        if (st == B3G_OK) {
            LeafArgs a;
            std::memset(&a, 0, sizeof a);
            a.in = p + (A - base) * kChunkBytes;
            a.len = (B - A) * kChunkBytes;
            a.n_chunks = a.n_full = B - A;
            a.counter_base = A;
            a.n_tiles = tiles;
            a.out = tile_cvs;
            a.status = status;
            a.wait_limit_ns = kWaitLimitNs;
            std::memcpy(a.key, h->kw, sizeof a.key);
            a.mode_flags = h->mode_flags;
            st = launch_leaf(a, kDefaultLeavesLog2, false, s);
        }
        if (st == B3G_OK) st = fork_aux(h, s);  // the tile CVs are ready
        RangesArgs ra;
        std::memset(&ra, 0, sizeof ra);
        ra.in = tile_cvs;
        ra.out = roots;
        std::memcpy(ra.key, h->kw, sizeof ra.key);
        ra.mode_flags = h->mode_flags;
        uint32_t nr = 0, widest = 1;
        for (size_t j : big) {
            if (st != B3G_OK) break;
            const uint64_t t0 = (pieces[j].pos - A) / tile, t = pieces[j].size / tile;
            if (t > 1024) {  // a very large piece: the ordinary multi-level reduction
                st = reduce_cvs_ws(tile_cvs + 32 * t0, t, h->kw, h->mode_flags, false, roots + 32 * j, huge, huge_ws, x);
                continue;
            }
            ra.start[nr] = static_cast<uint32_t>(t0);
            ra.count[nr] = static_cast<uint32_t>(t);
            ra.slot[nr] = static_cast<uint32_t>(j);
            widest = static_cast<uint32_t>(t) > widest ? static_cast<uint32_t>(t) : widest;
            ++nr;
        }
        if (st == B3G_OK && nr) {
            const unsigned threads = widest / 2 < 32 ? 32 : widest / 2;
            ranges_reduce_kernel<<<nr, threads, 0, x>>>(ra);
            e = cudaGetLastError();
            if (e != cudaSuccess) st = cuda_fail(e, "ranges_reduce_kernel launch");
        }
    }
    if (st == B3G_OK) {
        RecordArgs rec = record_args(h->state, h->kw, h->mode_flags, kRecPushMany);
        rec.depth = h->depth;
        rec.roots = roots;
        rec.npieces = static_cast<uint32_t>(pieces.size());
        uint32_t d = h->depth;
        for (size_t j = 0; j < pieces.size(); ++j) {
            rec.piece_pos[j] = pieces[j].pos;
            const uint32_t target = popcount64(pieces[j].pos);
            d = (d > target ? target : d) + 1;
        }
        st = launch_record(rec, x);
        if (st == B3G_OK) {
            h->depth = d;
            h->pushed = base + nchunks;
        }
    }
    e = cudaFreeAsync(scratch, x);
    if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "cudaFreeAsync");
    return st;
}

// A segment longer than acc while acc holds less than one chunk, on a hasher with the
// readers' stream, outside stream capture: the readers' stream assembles the boundary
// chunk (acc's bytes, then the segment's first `fill`) in a staging slot and, after the
// whole chunks have been pushed, copies the segment's last bytes into acc, so the
// caller's stream runs no copy of its own between two leaf launches.
b3g_status update_long(b3g_hasher *h, const uint8_t *p, uint64_t len, uint64_t fill, cudaStream_t s) {
    b3g_status st = B3G_OK;
    if (fill) {
        int slot = -1;
        st = stage_chunk_rd(h, h->acc, h->acc_len, p, fill, s, &slot);
        if (st == B3G_OK) st = push_record(h, h->slots + kChunkBytes * slot, slot);
        if (st != B3G_OK) return st;
        h->acc_len = 0;
    }
    const uint64_t full = (len - fill) / kChunkBytes;
    st = push_run(h, p + fill, full, s);
    if (st != B3G_OK) return st;
    const uint64_t tail = len - fill - full * kChunkBytes;
    if (tail) {
        st = fork_rd(h, s);
        const cudaError_t e = st == B3G_OK ? cudaMemcpyAsync(h->acc, p + fill + full * kChunkBytes, tail,
                                                             cudaMemcpyDeviceToDevice, h->rd)
                                           : cudaSuccess;
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
        if (st == B3G_OK) st = rd_handoff(h);
        if (st != B3G_OK) return st;
        h->acc_len = tail;
    }
    // the segment may be reused and acc read on `s` once the readers are done
    st = join_reads(h, s);
    if (st == B3G_OK) h->count += len;
    return st;
}

// Appends len bytes at p to acc (a copy on `s`).
b3g_status append_acc(b3g_hasher *h, const uint8_t *p, uint64_t len, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(h->acc + h->acc_len, p, len, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
    h->acc_len += len;
    return B3G_OK;
}

// Moves acc to an own kAccBytes buffer.  If the allocation fails the hasher keeps the
// 1024-byte buffer (and stops trying).
b3g_status grow_acc(b3g_hasher *h, cudaStream_t s) {
    uint8_t *bigger = nullptr;
    cudaError_t e = alloc_sync(reinterpret_cast<void **>(&bigger), kAccBytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        h->may_grow = false;
        return B3G_OK;
    }
    if (h->acc_len) {
        e = cudaMemcpyAsync(bigger, h->acc, h->acc_len, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) {
            cudaFree(bigger);
            return cuda_fail(e, "cudaMemcpyAsync");
        }
    }
    h->acc = bigger;
    h->acc_cap = kAccBytes;
    h->may_grow = false;
    return B3G_OK;
}

void hasher_clear(b3g_hasher *h) {
    h->count = h->pushed = 0;
    h->depth = 0;
    h->acc_len = 0;
}

}  // namespace

namespace {

// Extendable output of d_in[0..len) in the mode given by `key` (the key, or the IV)
// and `mode_flags`.
b3g_status xof_range(const void *d_in, uint64_t len, const uint8_t key[32], uint32_t mode_flags, uint8_t *d_out,
                     uint64_t out_len, cudaStream_t s) {
    uint32_t kw[8];
    key_words(key, kw);
    const uint64_t n = len == 0 ? 1 : ceil_div(len, kChunkBytes);
    uint64_t left_n = 1;
    while (n > 1 && left_n * 2 < n) left_n *= 2;
    const uint64_t left_bytes = left_n * kChunkBytes;
    // scratch: a state-shaped area for the record, then the two subtree workspaces
    const size_t ws_left = n > 1 ? blake3_workspace_size(left_bytes) : 0;
    const size_t ws_right = n > 1 ? blake3_workspace_size(len - left_bytes) : 0;
    const size_t off1 = (kStateBytes + 255) & ~size_t(255);
    const size_t off2 = off1 + ((ws_left + 255) & ~size_t(255));
    uint8_t *scratch = nullptr;
    cudaError_t e = alloc_async(reinterpret_cast<void **>(&scratch), off2 + ws_right, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync");
    uint32_t *rec = reinterpret_cast<uint32_t *>(scratch + kRecordOff);
    b3g_status st;
    if (n == 1) {
        RecordArgs ra = record_args(scratch, kw, mode_flags, kRecChunk);
        ra.in = static_cast<const uint8_t *>(d_in);
        ra.len = static_cast<uint32_t>(len);
        st = launch_record(ra, s);
    } else {
        // the root's children, written straight into the record's message words
        st = hash_range_ws(d_in, left_bytes, 0, key, mode_flags, false, reinterpret_cast<uint8_t *>(rec + 8),
                           scratch + off1, s);
        if (st == B3G_OK)
            st = hash_range_ws(static_cast<const uint8_t *>(d_in) + left_bytes, len - left_bytes, left_n, key,
                               mode_flags, false, reinterpret_cast<uint8_t *>(rec + 16), scratch + off2, s);
        if (st == B3G_OK) st = launch_record(record_args(scratch, kw, mode_flags, kRecParent), s);
    }
    if (st == B3G_OK) st = launch_xof(rec, d_out, out_len, s);
    e = cudaFreeAsync(scratch, s);
    if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "cudaFreeAsync");
    return st;
}

// A new hasher in the mode given by `key` (the key, or the IV) and `mode_flags`.
b3g_status hasher_create(const uint8_t key[32], uint32_t mode_flags, b3g_hasher **out) {
    *out = nullptr;
    b3g_hasher *h = new (std::nothrow) b3g_hasher;
    if (!h) return B3G_ERR_ARG;
    std::memcpy(h->key, key, 32);
    key_words(key, h->kw);
    h->mode_flags = mode_flags;
    hasher_clear(h);
    h->state = nullptr;
    cudaError_t e = cudaGetDevice(&h->device);
    if (e == cudaSuccess) e = alloc_sync(reinterpret_cast<void **>(&h->state), kStateBytes);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "hasher state");
    }
    h->acc = h->state + kBufOff;
    h->acc_cap = kChunkBytes;
    h->may_grow = true;
    const b3g_status st = streams_init(h, true);
    if (st != B3G_OK) {
        streams_release(h);
        cudaFree(h->state);
        delete h;
        return st;
    }
    *out = h;
    return B3G_OK;
}

// Digest of host bytes in the mode given by `key` (the key, or the IV) and
// `mode_flags`: copies into two staging slots overlap the hashing of the other slot.
b3g_status host_range(const void *h_in, uint64_t len, const uint8_t key[32], uint32_t mode_flags, uint8_t out32[32],
                      void *d_staging, size_t staging_bytes, b3g_stream_t stream) {
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t cs = nullptr;
    b3g_status st = cached_stream(0, &cs);
    if (st != B3G_OK) return st;
    constexpr size_t kSlotAlign = 1u << 20;
    constexpr size_t kHead = (kStateBytes + 255) & ~size_t(255);  // hasher state + digest
    if (d_staging && (reinterpret_cast<uintptr_t>(d_staging) & 255u)) return B3G_ERR_ALIGN;
    if (d_staging && staging_bytes < kHead + 2 * kSlotAlign) return B3G_ERR_WORKSPACE;
    bool own = false;
    if (!d_staging) {
        staging_bytes = kHead + 2 * (64u << 20);
        cudaError_t e = alloc_async(&d_staging, staging_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync");
        own = true;
    }
    const size_t slot = ((staging_bytes - kHead) / 2) & ~(kSlotAlign - 1);
    uint8_t *base = static_cast<uint8_t *>(d_staging);
    uint8_t *slots[2] = {base + kHead, base + kHead + slot};

    // a hasher whose state lives in the staging area; slot-sized segments bypass acc
    b3g_hasher h;
    std::memcpy(h.key, key, 32);
    key_words(key, h.kw);
    h.mode_flags = mode_flags;
    hasher_clear(&h);
    h.own_streams = h.read_pending = h.rd_pending = false;
    h.aux = h.rd = nullptr;
    h.ev_fork = h.ev_read = h.ev_done = nullptr;
    h.ev_fork_rd = h.ev_read_rd = h.ev_rd_done = h.ev_rd_all = nullptr;
    for (cudaEvent_t &ev : h.ev_slot) ev = nullptr;
    h.slots = nullptr;
    h.slot_next = 0;
    h.state = base;
    h.acc = base + kBufOff;
    h.acc_cap = kChunkBytes;
    h.may_grow = false;
    cudaError_t e = cudaGetDevice(&h.device);
    if (e != cudaSuccess) st = cuda_fail(e, "cudaGetDevice");
    if (st == B3G_OK) st = streams_init(&h, false);

    cudaEvent_t ev[5] = {};
    for (int i = 0; i < 5 && st == B3G_OK && e == cudaSuccess; ++i)
        e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    cudaEvent_t start = ev[0], copied[2] = {ev[1], ev[2]}, consumed[2] = {ev[3], ev[4]};
    if (st == B3G_OK && e == cudaSuccess) e = cudaEventRecord(start, s);  // staging is free from here on
    if (st == B3G_OK && e == cudaSuccess) e = cudaStreamWaitEvent(cs, start, 0);
    if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "event set-up");
    const uint8_t *src = static_cast<const uint8_t *>(h_in);
    uint64_t off = 0;
    for (uint64_t i = 0; st == B3G_OK && off < len; ++i) {
        const int b = static_cast<int>(i & 1);
        const uint64_t n = len - off < slot ? len - off : slot;
        if (i >= 2) e = cudaStreamWaitEvent(cs, consumed[b], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(slots[b], src + off, n, cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaEventRecord(copied[b], cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, copied[b], 0);
        if (e != cudaSuccess) {
            st = cuda_fail(e, "staging copy");
            break;
        }
        st = blake3_hasher_update(&h, slots[b], n, stream);
        if (st == B3G_OK && (e = cudaEventRecord(consumed[b], s)) != cudaSuccess) st = cuda_fail(e, "cudaEventRecord");
        off += n;
    }
    uint8_t *d_digest = base + kStateBytes;  // 32 bytes between the state and the slots
    if (st == B3G_OK) st = blake3_hasher_finalize(&h, d_digest, 32, stream);
    if (st == B3G_OK && (e = cudaMemcpyAsync(out32, d_digest, 32, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        st = cuda_fail(e, "cudaMemcpyAsync(digest)");
    if (h.aux && h.ev_done) join_all(&h, s);  // also after an error: nothing on the side stream outlives the staging
    if (own) {
        e = cudaFreeAsync(d_staging, s);
        if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "cudaFreeAsync");
    }
    e = cudaStreamSynchronize(s);
    if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "cudaStreamSynchronize");
    for (cudaEvent_t x : ev)
        if (x) cudaEventDestroy(x);
    streams_release(&h);
    return st;
}

}  // namespace

namespace {

// One gather launch: segments i, i+1, ... (up to K, skipping empty ones) while they fit
// in the accumulation buffer; advances i past them.  `launched` is false when segment
// i itself does not fit (nothing launched, i unchanged).
template <int K>
b3g_status gather_run(b3g_hasher *h, const void *const *d_ptrs, const uint64_t *lens, uint64_t count, uint64_t &i,
                      bool &launched, cudaStream_t s) {
    GatherArgs<K> ga;
    ga.dst = h->acc + h->acc_len;
    ga.n = 0;
    uint64_t bytes = 0, pieces = 0;
    while (i < count && ga.n < static_cast<uint32_t>(K) && h->acc_len + bytes + lens[i] <= h->acc_cap) {
        if (lens[i] > 0) {
            ga.src[ga.n] = static_cast<const uint8_t *>(d_ptrs[i]);
            ga.off[ga.n] = bytes;
            ga.len[ga.n] = lens[i];
            ga.piece0[ga.n] = static_cast<uint32_t>(pieces);
            pieces += (lens[i] + kGatherPiece - 1) / kGatherPiece;
            bytes += lens[i];
            ++ga.n;
        }
        ++i;
    }
    launched = ga.n > 0;
    if (!launched) return B3G_OK;
    ga.piece0[ga.n] = static_cast<uint32_t>(pieces);
    gather_kernel<K><<<static_cast<unsigned>(pieces), 256, 0, s>>>(ga);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "gather_kernel launch");
    h->acc_len += bytes;
    h->count += bytes;
    return B3G_OK;
}

}  // namespace

extern "C" {

b3g_status blake3_keyed_hash_xof(const void *d_in, uint64_t len, const uint8_t key[32], uint8_t *d_out,
                                 uint64_t out_len, b3g_stream_t stream) {
    if (!key || (!d_out && out_len > 0) || (!d_in && len > 0)) return B3G_ERR_NULL;
    return xof_range(d_in, len, key, kModeKeyed, d_out, out_len, reinterpret_cast<cudaStream_t>(stream));
}

b3g_status blake3_hash_xof(const void *d_in, uint64_t len, uint8_t *d_out, uint64_t out_len, b3g_stream_t stream) {
    if ((!d_out && out_len > 0) || (!d_in && len > 0)) return B3G_ERR_NULL;
    uint8_t iv[32];
    iv_key_bytes(iv);
    return xof_range(d_in, len, iv, kModeDefault, d_out, out_len, reinterpret_cast<cudaStream_t>(stream));
}



b3g_status blake3_hasher_new(const uint8_t key[32], b3g_hasher **out) {
    if (!key || !out) return B3G_ERR_NULL;
    return hasher_create(key, kModeKeyed, out);
}

b3g_status blake3_hasher_new_default(b3g_hasher **out) {
    if (!out) return B3G_ERR_NULL;
    uint8_t iv[32];
    iv_key_bytes(iv);
    return hasher_create(iv, kModeDefault, out);
}

void blake3_hasher_free(b3g_hasher *h) {
    if (!h) return;
    int prev = -1;
    if (cudaGetDevice(&prev) == cudaSuccess && prev != h->device) cudaSetDevice(h->device);
    streams_release(h);
    if (h->acc != h->state + kBufOff) cudaFree(h->acc);
    cudaFree(h->state);
    if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
    delete h;
}

b3g_status blake3_hasher_reset(b3g_hasher *h) {
    if (!h) return B3G_ERR_NULL;
    hasher_clear(h);
    return B3G_OK;
}

uint64_t blake3_hasher_count(const b3g_hasher *h) { return h ? h->count : 0; }

b3g_status blake3_hasher_update(b3g_hasher *h, const void *d_in, uint64_t len, b3g_stream_t stream) {
    if (!h || (!d_in && len > 0)) return B3G_ERR_NULL;
    if (len == 0) return B3G_OK;
    b3g_status st = check_device(h->device);
    if (st != B3G_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t *p = static_cast<const uint8_t *>(d_in);
    // under stream capture: no allocation outside the stream, and the side stream
    // rejoins completely, so that the captured graph is closed
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    if (h->acc_len + len > h->acc_cap && h->may_grow && !capturing && len < kAccBytes) {
        st = grow_acc(h, s);
        if (st != B3G_OK) return st;
    }
    // fits: keep the bytes (while the input is at most one chunk this is required, the
    // chunk may turn out to be the whole input and then needs ROOT)
    if (h->acc_len + len <= h->acc_cap) {
        st = append_acc(h, p, len, s);
        if (st == B3G_OK) h->count += len;
        return st;
    }
    if (h->rd && !capturing && h->acc_len < kChunkBytes) {
        const uint64_t fill = h->acc_len ? kChunkBytes - h->acc_len : 0;
        if (len - fill > h->acc_cap) return update_long(h, p, len, fill, s);
    }
    // more than acc holds, so more input follows every chunk in acc: complete its last
    // chunk, push all of acc, then push the segment's whole chunks if they do not fit
    // in acc either, and keep the rest
    uint64_t rest = len;
    const uint64_t fill_to = (kChunkBytes - h->acc_len % kChunkBytes) % kChunkBytes;
    const uint64_t fill = fill_to < rest ? fill_to : rest;
    if (fill) {
        st = append_acc(h, p, fill, s);
        if (st != B3G_OK) return st;
        p += fill;
        rest -= fill;
    }
    if (h->acc_len) {
        st = push_run(h, h->acc, h->acc_len / kChunkBytes, s);
        if (st != B3G_OK) return st;
        h->acc_len = 0;
    }
    if (rest > h->acc_cap) {
        const uint64_t full = rest / kChunkBytes;
        st = push_run(h, p, full, s);
        if (st != B3G_OK) return st;
        p += full * kChunkBytes;
        rest -= full * kChunkBytes;
    }
    // the side stream has read acc and the segment before `s` goes on
    st = capturing ? join_all(h, s) : join_reads(h, s);
    if (st != B3G_OK) return st;
    if (rest) {
        st = append_acc(h, p, rest, s);
        if (st != B3G_OK) return st;
    }
    h->count += len;
    return B3G_OK;
}


b3g_status blake3_hasher_update_many(b3g_hasher *h, const void *const *d_ptrs, const uint64_t *lens, uint64_t count,
                                     b3g_stream_t stream) {
    if (!h || (count > 0 && (!d_ptrs || !lens))) return B3G_ERR_NULL;
    for (uint64_t i = 0; i < count; ++i)
        if (!d_ptrs[i] && lens[i] > 0) return B3G_ERR_NULL;
    if (count == 0) return B3G_OK;
    b3g_status st = check_device(h->device);
    if (st != B3G_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    uint64_t i = 0;
    while (i < count) {
        if (lens[i] == 0) {
            ++i;
            continue;
        }
        if (h->acc_len + lens[i] > h->acc_cap && h->may_grow && cap == cudaStreamCaptureStatusNone &&
            lens[i] < kAccBytes) {
            st = grow_acc(h, s);
            if (st != B3G_OK) return st;
        }
        // the run of segments that fit in the accumulation buffer: one gather launch
        bool launched = false;
        st = count - i > static_cast<uint64_t>(kGatherSmall)
                 ? gather_run<kGatherBig>(h, d_ptrs, lens, count, i, launched, s)
                 : gather_run<kGatherSmall>(h, d_ptrs, lens, count, i, launched, s);
        if (st != B3G_OK) return st;
        if (!launched) {  // segment i does not fit: the ordinary update pushes what it must
            st = blake3_hasher_update(h, d_ptrs[i], lens[i], stream);
            if (st != B3G_OK) return st;
            ++i;
        }
    }
    return B3G_OK;
}

// Exported hasher state, little-endian: magic "B3GH", version, mode flags, stack depth,
// the key (or IV) bytes, bytes absorbed, chunks pushed, bytes buffered; then the stack
// (32 bytes per entry, bottom first) and the buffered bytes.
constexpr uint32_t kStateMagic = 0x48473342u;  // "B3GH"
constexpr uint32_t kStateVersion = 1;
constexpr size_t kStateHeader = 4 * 4 + 32 + 3 * 8;

size_t blake3_hasher_export_size(const b3g_hasher *h) {
    return h ? kStateHeader + 32ull * h->depth + h->acc_len : 0;
}

b3g_status blake3_hasher_export(const b3g_hasher *h, void *h_buf, size_t buf_bytes, b3g_stream_t stream) {
    if (!h || !h_buf) return B3G_ERR_NULL;
    if (buf_bytes < blake3_hasher_export_size(h)) return B3G_ERR_WORKSPACE;
    b3g_status st = check_device(h->device);
    if (st != B3G_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    b3g_hasher t = *h;
    st = join_all(&t, s);  // the stack is complete on `s`
    if (st != B3G_OK) return st;
    uint8_t *out = static_cast<uint8_t *>(h_buf);
    const uint32_t words[4] = {kStateMagic, kStateVersion, h->mode_flags, h->depth};
    const uint64_t counts[3] = {h->count, h->pushed, h->acc_len};
    std::memcpy(out, words, sizeof words);
    std::memcpy(out + 16, h->key, 32);
    std::memcpy(out + 48, counts, sizeof counts);
    cudaError_t e = cudaSuccess;
    if (h->depth) e = cudaMemcpyAsync(out + kStateHeader, h->state, 32ull * h->depth, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && h->acc_len)
        e = cudaMemcpyAsync(out + kStateHeader + 32ull * h->depth, h->acc, h->acc_len, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "hasher export");
}

b3g_status blake3_hasher_import(const void *h_buf, size_t buf_bytes, b3g_hasher **out, b3g_stream_t stream) {
    if (!h_buf || !out) return B3G_ERR_NULL;
    *out = nullptr;
    if (buf_bytes < kStateHeader) return B3G_ERR_ARG;
    const uint8_t *in = static_cast<const uint8_t *>(h_buf);
    uint32_t words[4];
    uint64_t counts[3];
    uint8_t key[32];
    std::memcpy(words, in, sizeof words);
    std::memcpy(key, in + 16, 32);
    std::memcpy(counts, in + 48, sizeof counts);
    const uint32_t mode_flags = words[2], depth = words[3];
    const uint64_t count = counts[0], pushed = counts[1], acc_len = counts[2];
    // the record must describe a state update() can reach
    if (words[0] != kStateMagic || words[1] != kStateVersion) return B3G_ERR_ARG;
    if (mode_flags != kModeKeyed && mode_flags != kModeDefault) return B3G_ERR_ARG;
    if (depth > kStackSlots - 1 || acc_len > kAccBytes || pushed > (1ull << 53)) return B3G_ERR_ARG;
    if (count != pushed * kChunkBytes + acc_len || (pushed == 0) != (depth == 0)) return B3G_ERR_ARG;
    if (pushed > 0 && count <= kChunkBytes) return B3G_ERR_ARG;
    if (buf_bytes < kStateHeader + 32ull * depth + acc_len) return B3G_ERR_ARG;

    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    b3g_hasher *h = nullptr;
    b3g_status st = hasher_create(key, mode_flags, &h);
    if (st != B3G_OK) return st;
    if (acc_len > h->acc_cap) {
        st = grow_acc(h, s);
        if (st == B3G_OK && acc_len > h->acc_cap) st = cuda_fail(cudaErrorMemoryAllocation, "hasher import buffer");
    }
    cudaError_t e = cudaSuccess;
    if (st == B3G_OK && depth)
        e = cudaMemcpyAsync(h->state, in + kStateHeader, 32ull * depth, cudaMemcpyHostToDevice, s);
    if (st == B3G_OK && e == cudaSuccess && acc_len)
        e = cudaMemcpyAsync(h->acc, in + kStateHeader + 32ull * depth, acc_len, cudaMemcpyHostToDevice, s);
    if (st == B3G_OK && e == cudaSuccess) e = cudaStreamSynchronize(s);  // the caller may free h_buf
    if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "hasher import");
    if (st != B3G_OK) {
        blake3_hasher_free(h);
        return st;
    }
    h->count = count;
    h->pushed = pushed;
    h->depth = depth;
    h->acc_len = acc_len;
    *out = h;
    return B3G_OK;
}

b3g_status blake3_keyed_hash_host(const void *h_in, uint64_t len, const uint8_t key[32], uint8_t out32[32],
                                  void *d_staging, size_t staging_bytes, b3g_stream_t stream) {
    if (!key || !out32 || (!h_in && len > 0)) return B3G_ERR_NULL;
    return host_range(h_in, len, key, kModeKeyed, out32, d_staging, staging_bytes, stream);
}

b3g_status blake3_hash_host(const void *h_in, uint64_t len, uint8_t out32[32], void *d_staging,
                            size_t staging_bytes, b3g_stream_t stream) {
    if (!out32 || (!h_in && len > 0)) return B3G_ERR_NULL;
    uint8_t iv[32];
    iv_key_bytes(iv);
    return host_range(h_in, len, iv, kModeDefault, out32, d_staging, staging_bytes, stream);
}

b3g_status blake3_hasher_finalize(const b3g_hasher *hc, uint8_t *d_out, uint64_t out_len, b3g_stream_t stream) {
    if (!hc || (!d_out && out_len > 0)) return B3G_ERR_NULL;
    b3g_status st = check_device(hc->device);
    if (st != B3G_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // a working copy: chunks still in acc are pushed onto a scratch copy of the stack,
    // so the hasher itself is unchanged
    b3g_hasher t = *hc;
    st = join_all(&t, s);
    if (st != B3G_OK) return st;
    if (t.count <= kChunkBytes) {
        RecordArgs ra = record_args(t.state, t.kw, t.mode_flags, kRecChunk);
        ra.in = t.acc;
        ra.len = static_cast<uint32_t>(t.count);
        st = launch_record(ra, s);
        if (st != B3G_OK) return st;
        return launch_xof(reinterpret_cast<const uint32_t *>(t.state + kRecordOff), d_out, out_len, s);
    }
    // every chunk of acc but the last is pushed; the last (1..1024 bytes) is finished by
    // the record launch
    const uint64_t k = t.acc_len ? (t.acc_len - 1) / kChunkBytes : 0;
    uint8_t *scratch = nullptr;
    cudaError_t e;
    if (k) {
        e = alloc_async(reinterpret_cast<void **>(&scratch), kStateBytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync");
        if (t.depth) e = cudaMemcpyAsync(scratch, t.state, 32ull * t.depth, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) st = cuda_fail(e, "cudaMemcpyAsync");
        t.state = scratch;
        if (st == B3G_OK) st = push_run(&t, t.acc, k, s);
        const b3g_status js = join_all(&t, s);
        if (st == B3G_OK) st = js;
    }
    if (st == B3G_OK) {
        RecordArgs ra = record_args(t.state, t.kw, t.mode_flags, kRecFinalize);
        ra.in = t.acc + k * kChunkBytes;
        ra.len = static_cast<uint32_t>(t.acc_len - k * kChunkBytes);
        ra.depth = t.depth;
        ra.pushed = t.pushed;
        st = launch_record(ra, s);
    }
    if (st == B3G_OK) st = launch_xof(reinterpret_cast<const uint32_t *>(t.state + kRecordOff), d_out, out_len, s);
    if (scratch) {
        e = cudaFreeAsync(scratch, s);
        if (st == B3G_OK && e != cudaSuccess) st = cuda_fail(e, "cudaFreeAsync");
    }
    return st;
}

}  // extern "C"

// b3g_reduce.cu -- reduction of subtree CVs to the root, and the bounded-wait probe.
//
// Source page: "BLAKE3 GPU 400x faster hashing" (qfminer.top), section
// "Kernel 2 和 3": after the leaf kernel every CTA has produced one 32-byte subtree
// root; a second kernel loads a group of those roots into shared memory and reduces
// it with the same routine, setting ROOT on the final compression when one group is
// left; a third, single-CTA kernel finishes when more than one group remains.
//
// Here one kernel serves every level: the host relaunches it on its own output until
// one CV is left, and the launch with a single group sets ROOT.  Groups are aligned
// runs of 2^g CVs, so every group but the last is a perfect subtree of the tree and
// the last one folds right to left (block_tree), which keeps the result identical
// to the tree of the whole input.
#include <mutex>

#include "b3g_device.cuh"
#include "b3g_internal.h"

namespace b3g {

constexpr uint32_t kBarReduce = 1;
constexpr int kReduceMaxThreads = 512;

__global__ void __launch_bounds__(kReduceMaxThreads) reduce_cvs_kernel(const ReduceArgs a) {
    __shared__ __align__(128) uint8_t node_mem[kReduceMaxThreads * 32];
    // launched early behind the kernel that writes a.in: wait for its results, and let
    // the next level's launch start early in turn
    grid_dependency_wait();
    launch_dependents();
    const uint32_t nodes = smem_u32(node_mem);
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = a.key[i];
    const uint32_t tid = threadIdx.x;
    const uint32_t nthreads = blockDim.x;
    const bool final_group = a.root && gridDim.x == 1;

    const uint64_t first = static_cast<uint64_t>(blockIdx.x) * a.group;
    const uint64_t rem = a.count - first;
    const uint32_t m = rem < a.group ? static_cast<uint32_t>(rem) : a.group;

    // first level straight from global memory: CVs 2*tid and 2*tid+1 are 64
    // contiguous bytes
    const uint32_t half = m >> 1;
    uint32_t res[8];
    bool have = false;
    if (tid < half) {
        const uint4 *p = reinterpret_cast<const uint4 *>(a.in + (first + 2ull * tid) * 32);
        uint4 w0 = p[0], w1 = p[1], w2 = p[2], w3 = p[3];
        uint32_t l[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t r[8] = {w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
        parent(key, a.mode_flags, l, r, final_group && m == 2, res);
        have = true;
    } else if (tid == half && (m & 1u)) {
        const uint4 *p = reinterpret_cast<const uint4 *>(a.in + (first + m - 1) * 32);
        uint4 w0 = p[0], w1 = p[1];
        res[0] = w0.x; res[1] = w0.y; res[2] = w0.z; res[3] = w0.w;
        res[4] = w1.x; res[5] = w1.y; res[6] = w1.z; res[7] = w1.w;
        have = true;
    }
    if (have) store_node(nodes, tid, res);
    named_bar_sync(kBarReduce, nthreads);
    uint32_t out[8];
    block_tree(nodes, (m + 1) >> 1, tid, nthreads, kBarReduce, key, a.mode_flags, final_group, out);
    if (tid == 0) {
        uint4 *o = reinterpret_cast<uint4 *>(a.out + static_cast<uint64_t>(blockIdx.x) * 32);
        o[0] = make_uint4(out[0], out[1], out[2], out[3]);
        o[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
}

// One thread waits on a barrier that nothing ever completes; the bounded wait
// must give up and report it.
__global__ void wait_probe_kernel(uint64_t limit_ns, int *flag) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const bool done = mbar_wait_bounded(b, 0, limit_ns);
    *flag = done ? 0 : 1;
}

// The same probe reporting in a caller's status word: B3G_DEVICE_STATUS_TIMEOUT is ORed
// into *status when the wait gives up, in stream order, as the hashing kernels do.
__global__ void wait_probe_status_kernel(uint64_t limit_ns, uint32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(b, 0, limit_ns)) atomicOr(status, B3G_DEVICE_STATUS_TIMEOUT);
}

// Compression-only loop: every thread runs `iters` chained compressions of the hashing
// kernels' compress() with its message held in registers (fed back from the CV so that
// nothing is hoisted) and no memory traffic; the ceiling the leaf kernel is measured
// against.  The sink is written only on an impossible value, to keep the result live.
__global__ void __launch_bounds__(128) compress_rate_kernel(uint32_t seed, uint32_t iters, uint32_t *sink) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t cv[8], m[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) cv[i] = seed ^ (t * 0x9E3779B9u + static_cast<uint32_t>(i));
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = seed + t * 16u + static_cast<uint32_t>(i);
#pragma unroll 1
    for (uint32_t it = 0; it < iters; ++it) {
        compress(cv, m, it, 0u, kBlockLen, kModeKeyed);
        m[0] ^= cv[0];
        m[5] ^= cv[3];
    }
    if ((cv[0] ^ cv[7]) == 0x5EED5EEDu && cv[1] == seed) *sink = cv[2];
}

// ---------------------------------------------------------------------------------
// Several lanes per chunk (page section "未来工作": several threads could hash the same
// chunk).  One compression spread over the 4 lanes of an aligned group of 4: lane q
// holds column q of the state, v[q], v[4 + q], v[8 + q], v[12 + q].  The column step is
// one G per lane; for the diagonal step rows 1, 2 and 3 are rotated by 1, 2 and 3 lanes
// with shuffles, each lane runs one G, and the rows are rotated back.  w[r] holds the
// lane's message words of round r (column x, y, diagonal x, y).  The output CV words q
// and 4 + q stay on lane q, where the next compression of a chain takes them.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void compress_4lane(uint32_t &cva, uint32_t &cvb, const uint32_t w[7][4], uint32_t q,
                                               uint32_t counter_lo, uint32_t counter_hi, uint32_t block_len,
                                               uint32_t flags) {
    uint32_t a = cva, b = cvb;
    uint32_t c = q == 0 ? kIv0 : q == 1 ? kIv1 : q == 2 ? kIv2 : kIv3;
    uint32_t d = q == 0 ? counter_lo : q == 1 ? counter_hi : q == 2 ? block_len : flags;
    const uint32_t up1 = (q + 1) & 3u, up2 = (q + 2) & 3u, up3 = (q + 3) & 3u;
#pragma unroll
    for (int r = 0; r < 7; ++r) {
        g<0>(a, b, c, d, w[r][0], w[r][1]);
        b = __shfl_sync(0xffffffffu, b, up1, 4);
        c = __shfl_sync(0xffffffffu, c, up2, 4);
        d = __shfl_sync(0xffffffffu, d, up3, 4);
        g<4>(a, b, c, d, w[r][2], w[r][3]);
        b = __shfl_sync(0xffffffffu, b, up3, 4);
        c = __shfl_sync(0xffffffffu, c, up2, 4);
        d = __shfl_sync(0xffffffffu, d, up1, 4);
    }
    cva = a ^ c;
    cvb = b ^ d;
}

// The message words lane Q of a group of 4 needs in each round.
template <int Q>
__device__ __forceinline__ void lane_words(const uint32_t m[16], uint32_t w[7][4]) {
#pragma unroll
    for (int r = 0; r < 7; ++r) {
        w[r][0] = m[msg_index(r, 2 * Q)];
        w[r][1] = m[msg_index(r, 2 * Q + 1)];
        w[r][2] = m[msg_index(r, 8 + 2 * Q)];
        w[r][3] = m[msg_index(r, 9 + 2 * Q)];
    }
}

// Latency of a chain of `chain` dependent keyed compressions in one warp: L = 1, one
// chain per lane (32 chains, the hashing kernels' compress); L = 4, one chain per group
// of 4 lanes (8 chains, compress_4lane).  Chain g starts from the key, compresses the
// message m[i] = (16 g + i) * 0x9E3779B9 (mod 2^32) at counter j in step j, with block
// length 64 and flags KEYED_HASH, and writes its final CV to out + 32 g.  Lane 0 writes
// the clock cycles of the whole chain to *cycles.
template <int L>
__global__ void __launch_bounds__(32) compress_latency_kernel(uint32_t chain, const LatencyArgs a) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t gid = lane / L;
    uint32_t m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = (16u * gid + static_cast<uint32_t>(i)) * 0x9E3779B9u;
    long long t0, t1;
    if constexpr (L == 1) {
        uint32_t cv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[i] = a.key[i];
        __syncwarp();
        t0 = clock64();
#pragma unroll 1
        for (uint32_t j = 0; j < chain; ++j) compress(cv, m, j, 0u, kBlockLen, kModeKeyed);
        t1 = clock64();
        uint4 *o = reinterpret_cast<uint4 *>(a.out + 32ull * gid);
        o[0] = make_uint4(cv[0], cv[1], cv[2], cv[3]);
        o[1] = make_uint4(cv[4], cv[5], cv[6], cv[7]);
    } else {
        const uint32_t q = lane & 3u;
        uint32_t w[7][4];
        switch (q) {
            case 0: lane_words<0>(m, w); break;
            case 1: lane_words<1>(m, w); break;
            case 2: lane_words<2>(m, w); break;
            default: lane_words<3>(m, w); break;
        }
        uint32_t cva = a.key[q], cvb = a.key[4 + q];
        __syncwarp();
        t0 = clock64();
#pragma unroll 1
        for (uint32_t j = 0; j < chain; ++j) compress_4lane(cva, cvb, w, q, j, 0u, kBlockLen, kModeKeyed);
        t1 = clock64();
        uint32_t *o = reinterpret_cast<uint32_t *>(a.out + 32ull * gid);
        o[q] = cva;
        o[4 + q] = cvb;
    }
    if (lane == 0) *a.cycles = static_cast<unsigned long long>(t1 - t0);
}

b3g_status launch_compress_latency(int lanes, uint32_t chain, const LatencyArgs &a, cudaStream_t stream) {
    if (lanes == 1)
        compress_latency_kernel<1><<<1, 32, 0, stream>>>(chain, a);
    else if (lanes == 4)
        compress_latency_kernel<4><<<1, 32, 0, stream>>>(chain, a);
    else
        return B3G_ERR_ARG;
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "compress_latency_kernel launch");
}

b3g_status launch_compress_rate(uint32_t blocks, uint32_t iters, uint32_t *d_sink, cudaStream_t stream) {
    compress_rate_kernel<<<blocks, 128, 0, stream>>>(0x2545F491u, iters, d_sink);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "compress_rate_kernel launch");
}

// Sets one device word to zero in stream order.  A kernel launched with programmatic
// stream serialization, unlike a memset, lets the launch behind it (the leaf kernel,
// which waits for this grid in griddepcontrol.wait before it touches the word) start
// early; and it waits itself for the kernel ahead, which may still use the word (an
// earlier call on the same workspace).
__global__ void __launch_bounds__(32) zero_word_kernel(uint32_t *p) {
    grid_dependency_wait();
    if (threadIdx.x == 0) *p = 0u;
    launch_dependents();
}

b3g_status launch_zero_word(uint32_t *p, cudaStream_t stream) {
    const cudaError_t e = launch_pdl(zero_word_kernel, dim3(1), dim3(32), 0, stream, p);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "zero_word_kernel launch");
}

b3g_status launch_reduce(const ReduceArgs &a, cudaStream_t stream) {
    if (a.count == 0 || a.group < 2 || a.group > 2 * kReduceMaxThreads || (a.group & (a.group - 1)) != 0)
        return B3G_ERR_ARG;
    const uint64_t groups = (a.count + a.group - 1) / a.group;
    if (groups > 0x7fffffffull) return B3G_ERR_ARG;
    const int threads = a.group / 2 < 32 ? 32 : static_cast<int>(a.group / 2);
    // the launch overlaps the tail of the kernel ahead (the leaf kernel or the previous
    // level), whose output it waits for
    cudaError_t e = launch_pdl(reduce_cvs_kernel, dim3(static_cast<unsigned>(groups)),
                               dim3(static_cast<unsigned>(threads)), 0, stream, a);
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "reduce_cvs_kernel launch");
}

b3g_status launch_wait_probe(uint64_t limit_ns, int *d_flag, cudaStream_t stream) {
    wait_probe_kernel<<<1, 1, 0, stream>>>(limit_ns, d_flag);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "wait_probe_kernel launch");
}

b3g_status launch_wait_probe_status(uint64_t limit_ns, uint32_t *d_status, cudaStream_t stream) {
    wait_probe_status_kernel<<<1, 1, 0, stream>>>(limit_ns, d_status);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "wait_probe_status_kernel launch");
}

}  // namespace b3g

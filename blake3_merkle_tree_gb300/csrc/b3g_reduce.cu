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

b3g_status launch_compress_rate(uint32_t blocks, uint32_t iters, uint32_t *d_sink, cudaStream_t stream) {
    compress_rate_kernel<<<blocks, 128, 0, stream>>>(0x2545F491u, iters, d_sink);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? B3G_OK : cuda_fail(e, "compress_rate_kernel launch");
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

}  // namespace b3g

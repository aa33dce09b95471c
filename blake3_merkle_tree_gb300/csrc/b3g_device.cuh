// b3g_device.cuh -- device building blocks for the keyed BLAKE3 kernels (sm_103a).
//
// Source page: "BLAKE3 GPU 400x faster hashing" (qfminer.top).
//   section "压缩函数": one thread compresses one chunk entirely in registers, the
//     round function fully unrolled; 16 chained compressions per chunk, CHUNK_START
//     on the first block and CHUNK_END on the last; the key is the initial CV.
//   section "Merkle Tree 归约": parent = compress(key, left || right, counter 0,
//     length 64, KEYED_HASH | PARENT); halving levels with a barrier between them;
//     non-power-of-two leaf counts fold the binary decomposition right to left.
//   section "未来工作": exchange CVs between threads with warp primitives instead
//     of shared memory during the reduction.
// Round constants follow the BLAKE3 specification (O'Connor et al., 2020).
#pragma once

#include <cstdint>

namespace b3g {

// ---------------------------------------------------------------------------------
// Constants of the BLAKE3 specification.
// ---------------------------------------------------------------------------------
constexpr uint32_t kChunkLen = 1024;
constexpr uint32_t kBlockLen = 64;

constexpr uint32_t kIv0 = 0x6A09E667u, kIv1 = 0xBB67AE85u, kIv2 = 0x3C6EF372u, kIv3 = 0xA54FF53Au;

constexpr uint32_t kChunkStart = 1u, kChunkEnd = 2u, kParent = 4u, kRoot = 8u, kKeyedHash = 16u;

// Message word that G-slot i reads in round r: the message is permuted between
// rounds by P (word i of the next round is word P[i] of this one), so round r
// reads original word P^r(i).  Evaluated at compile time; with the rounds fully
// unrolled the permutation is pure register renaming.
__host__ __device__ constexpr int msg_index(int round, int slot) {
    constexpr int P[16] = {2, 6, 3, 10, 7, 0, 4, 13, 1, 11, 12, 5, 9, 14, 15, 8};
    int i = slot;
    for (int r = 0; r < round; ++r) i = P[i];
    return i;
}

// ---------------------------------------------------------------------------------
// Rotations: byte permutes for 16 and 8, funnel shifts for 12 and 7.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t rotr16(uint32_t x) { return __byte_perm(x, 0, 0x1032); }
__device__ __forceinline__ uint32_t rotr8(uint32_t x) { return __byte_perm(x, 0, 0x0321); }
__device__ __forceinline__ uint32_t rotr12(uint32_t x) { return __funnelshift_r(x, x, 12); }
__device__ __forceinline__ uint32_t rotr7(uint32_t x) { return __funnelshift_r(x, x, 7); }

// Additions of G.  On GB300 the XORs (LOP3), byte permutes (PRMT), funnel shifts
// (SHF) and three-input adds (IADD3) issue on the 16-lane ALU pipe, integer
// multiply-adds (IMAD) on the separate 16-lane FMA pipe.  Form 3 (the default)
// computes each three-input add a + b + x as two IMADs x * 1 + a, b * 1 + t with the
// multiplier 1 read from constant memory, so the compiler cannot fold them back into
// an IADD3; it already issues the two-input adds c + d as IMAD by itself.  A G is then
// 8 ALU instructions (4 XOR, 4 rotates) + 6 FMA instead of 10 + 2.  Measured on the
// leaf kernel (1 GiB, ncu): 11.0 -> 8.9 ALU and 2.3 -> 6.5 FMA warp instructions per
// G, 731 -> 606 us.  Form 0 leaves every add to the compiler, form 1 also forces the
// two-input adds through the constant 1 (slower: 657 us), form 2 writes the multiplier
// as an immediate (the compiler turns it back into IADD3).
#ifndef B3G_G_FORM
#define B3G_G_FORM 3
#endif

static __constant__ uint32_t c_one = 1u;

__device__ __forceinline__ uint32_t imad_add(uint32_t x, uint32_t y) {
    uint32_t r;
#if B3G_G_FORM == 2
    asm("mad.lo.u32 %0, %1, 1, %2;" : "=r"(r) : "r"(x), "r"(y));
#else
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(c_one), "r"(y));
#endif
    return r;
}

// a + b + x (x a message word: added first, it does not wait for b)
__device__ __forceinline__ uint32_t add3(uint32_t a, uint32_t b, uint32_t x) {
#if B3G_G_FORM == 0
    return a + b + x;
#else
    return imad_add(b, imad_add(x, a));
#endif
}

__device__ __forceinline__ uint32_t add2(uint32_t c, uint32_t d) {
#if B3G_G_FORM == 0 || B3G_G_FORM == 3
    return c + d;
#else
    return imad_add(d, c);
#endif
}

// Rotations on the FMA pipe.  x * 2^k as a 64-bit product holds x << k in its low
// word and x >> (32 - k) in its high word; the two share no bit, so their sum is the
// rotation left by k (right by 32 - k): one multiply (low word) and one multiply-add
// (high word plus the low word).  The multiplier comes from constant memory, so the
// compiler keeps the multiplies instead of turning them into shifts.  Bit j of
// B3G_ROT_FMA (G number j of a round: 0-3 columns, 4-7 diagonals) moves that G's
// rotation by 7 to the FMA pipe, bit 8 + j its rotation by 12; 0 keeps every rotation
// on the ALU pipe.
#ifndef B3G_ROT_FMA
#define B3G_ROT_FMA 0
#endif

static __constant__ uint32_t c_pow25 = 1u << 25;  // rotation right by 7
static __constant__ uint32_t c_pow20 = 1u << 20;  // rotation right by 12

__device__ __forceinline__ uint32_t rotr_fma(uint32_t x, uint32_t pow) {
    uint32_t lo, r;
    asm("mul.lo.u32 %0, %1, %2;" : "=r"(lo) : "r"(x), "r"(pow));
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(pow), "r"(lo));
    return r;
}

template <int J>
__device__ __forceinline__ void g(uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d, uint32_t x,
                                  uint32_t y) {
    constexpr bool kFma7 = (B3G_ROT_FMA >> J) & 1, kFma12 = (B3G_ROT_FMA >> (8 + J)) & 1;
    a = add3(a, b, x);
    d = rotr16(d ^ a);
    c = add2(c, d);
    b = kFma12 ? rotr_fma(b ^ c, c_pow20) : rotr12(b ^ c);
    a = add3(a, b, y);
    d = rotr8(d ^ a);
    c = add2(c, d);
    b = kFma7 ? rotr_fma(b ^ c, c_pow25) : rotr7(b ^ c);
}

template <int R>
__device__ __forceinline__ void round_fn(uint32_t v[16], const uint32_t m[16]) {
    // columns
    g<0>(v[0], v[4], v[8], v[12], m[msg_index(R, 0)], m[msg_index(R, 1)]);
    g<1>(v[1], v[5], v[9], v[13], m[msg_index(R, 2)], m[msg_index(R, 3)]);
    g<2>(v[2], v[6], v[10], v[14], m[msg_index(R, 4)], m[msg_index(R, 5)]);
    g<3>(v[3], v[7], v[11], v[15], m[msg_index(R, 6)], m[msg_index(R, 7)]);
    // diagonals
    g<4>(v[0], v[5], v[10], v[15], m[msg_index(R, 8)], m[msg_index(R, 9)]);
    g<5>(v[1], v[6], v[11], v[12], m[msg_index(R, 10)], m[msg_index(R, 11)]);
    g<6>(v[2], v[7], v[8], v[13], m[msg_index(R, 12)], m[msg_index(R, 13)]);
    g<7>(v[3], v[4], v[9], v[14], m[msg_index(R, 14)], m[msg_index(R, 15)]);
}

// One compression; cv (8 words) is replaced by the first 8 output words.
__device__ __forceinline__ void compress(uint32_t cv[8], const uint32_t m[16], uint32_t counter_lo,
                                         uint32_t counter_hi, uint32_t block_len, uint32_t flags) {
    uint32_t v[16] = {cv[0], cv[1], cv[2],      cv[3],      cv[4],     cv[5], cv[6], cv[7],
                      kIv0,  kIv1,  kIv2,       kIv3,       counter_lo, counter_hi, block_len, flags};
    round_fn<0>(v, m);
    round_fn<1>(v, m);
    round_fn<2>(v, m);
    round_fn<3>(v, m);
    round_fn<4>(v, m);
    round_fn<5>(v, m);
    round_fn<6>(v, m);
#pragma unroll
    for (int i = 0; i < 8; ++i) cv[i] = v[i] ^ v[i + 8];
}

// One compression keeping all 16 output words (extendable output): words 0..7 are
// v[i] ^ v[i+8], words 8..15 are v[i+8] ^ cv[i].
__device__ __forceinline__ void compress_full(const uint32_t cv[8], const uint32_t m[16], uint32_t counter_lo,
                                              uint32_t counter_hi, uint32_t block_len, uint32_t flags,
                                              uint32_t out[16]) {
    uint32_t v[16] = {cv[0], cv[1], cv[2],      cv[3],      cv[4],     cv[5], cv[6], cv[7],
                      kIv0,  kIv1,  kIv2,       kIv3,       counter_lo, counter_hi, block_len, flags};
    round_fn<0>(v, m);
    round_fn<1>(v, m);
    round_fn<2>(v, m);
    round_fn<3>(v, m);
    round_fn<4>(v, m);
    round_fn<5>(v, m);
    round_fn<6>(v, m);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        out[i] = v[i] ^ v[i + 8];
        out[i + 8] = v[i + 8] ^ cv[i];
    }
}

// Parent node: key as CV, left || right as the message.  `mode_flags` is the flag bit
// every compression of the hash mode carries: KEYED_HASH in keyed mode, none in the
// default mode (whose `key` is the IV).
__device__ __forceinline__ void parent(const uint32_t key[8], uint32_t mode_flags, const uint32_t l[8],
                                       const uint32_t r[8], bool root, uint32_t out[8]) {
    uint32_t m[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m[i] = l[i];
        m[i + 8] = r[i];
    }
    uint32_t cv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cv[i] = key[i];
    compress(cv, m, 0u, 0u, kBlockLen, mode_flags | kParent | (root ? kRoot : 0u));
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = cv[i];
}

// ---------------------------------------------------------------------------------
// Shared-memory, barrier and bulk-tensor-copy primitives (inline PTX).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test with a suspend-time hint: a thread whose phase has not completed may be
// suspended until it completes or about `hint_ns` nanoseconds have passed, instead of
// returning at once to poll again.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Suspend-time hint of the bounded waits (0: none, the hardware's own limit).  Without
// it the reducer warp, idle most of the time, polls its barrier and takes issue slots
// from the consumers; with a hint it sleeps until the phase completes.  Measured (leaf
// kernel, GB/s): 12 GiB + 777 B 2223 -> 2261, 4 GiB 2180 -> 2219, 256 MiB 1839 -> 1859,
// the same with 1 us and 20 us.
#ifndef B3G_WAIT_HINT_NS
#define B3G_WAIT_HINT_NS 20000
#endif

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the barrier phase with the given parity has completed, or give up
// after limit_ns nanoseconds.  Returns false if it gave up.  Every wait in the
// hashing kernels goes through here, so no kernel can spin forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#if B3G_WAIT_HINT_NS
        if (mbar_try_wait_hint(bar, parity, B3G_WAIT_HINT_NS)) return true;
#else
        if (mbar_try_wait(bar, parity)) return true;
#endif
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// 2-D tiled bulk tensor copy global -> shared, completion signalled on `bar`
// through the transaction count.  x is the innermost (word) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 16-byte asynchronous copy global -> shared (cached in L2 only), tracked per thread in
// copy groups; the L2 fetches the whole 256-byte segment around it, so the next blocks
// of the same chunk are L2 hits.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Closes this thread's current copy group (an empty group if it issued no copy).
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Waits until at most N of this thread's copy groups are still in flight.  The copies
// of the completed groups are then visible to this thread; a barrier makes them
// visible to the others.  A hardware wait for the thread's own copies, not a spin.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before its later
// async-proxy ones (a bulk copy into a stage the warp has just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch.  A grid launched with programmatic stream
// serialization may start before the grid ahead of it in the stream has finished;
// grid_dependency_wait() returns once that grid has completed and its memory writes
// are visible (at once if there is none).  launch_dependents() lets the grid behind
// this one start early (its CTAs then wait in grid_dependency_wait()).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over `nthreads` threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t res;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(res)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return res != 0;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint64_t lds64(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void sts64(uint32_t addr, uint64_t v) {
    asm volatile("st.shared.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------------
// Loads of one 64-byte block straight from global memory, for the partial last
// chunk and for inputs that cannot use the bulk tensor copy.  Bytes at or beyond
// `len` read as zero, and no byte outside [base, base + len) is touched.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t load_byte(const uint8_t *base, uint64_t len, uint64_t off) {
    return off < len ? static_cast<uint32_t>(__ldg(base + off)) : 0u;
}

__device__ __forceinline__ void load_block_global(const uint8_t *base, uint64_t len, uint64_t off,
                                                  uint32_t m[16]) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(base) + off;
    if (off + kBlockLen <= len && (addr & 15u) == 0) {
        const uint4 *p = reinterpret_cast<const uint4 *>(base + off);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 w = __ldg(p + q);
            m[4 * q + 0] = w.x;
            m[4 * q + 1] = w.y;
            m[4 * q + 2] = w.z;
            m[4 * q + 3] = w.w;
        }
        return;
    }
    const uintptr_t lo = addr & ~static_cast<uintptr_t>(3);
    const uintptr_t hi = (addr + kBlockLen + 3) & ~static_cast<uintptr_t>(3);
    const uintptr_t buf_lo = reinterpret_cast<uintptr_t>(base);
    const uintptr_t buf_hi = buf_lo + len;
    if (lo >= buf_lo && hi <= buf_hi) {
        // every aligned word covering the block lies inside the buffer
        const uint32_t *w = reinterpret_cast<const uint32_t *>(lo);
        const uint32_t sh = static_cast<uint32_t>(addr & 3u) * 8u;
        uint32_t prev = __ldg(w);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            uint32_t next = (sh == 0 && i == 15) ? 0u : __ldg(w + i + 1);
            m[i] = sh == 0 ? prev : __funnelshift_r(prev, next, sh);
            prev = next;
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint64_t o = off + 4u * i;
        m[i] = load_byte(base, len, o) | (load_byte(base, len, o + 1) << 8) |
               (load_byte(base, len, o + 2) << 16) | (load_byte(base, len, o + 3) << 24);
    }
}

// The same block load for the plain-load kernel, which reads every block of an input
// that is not 16-byte aligned: when the five 16-byte units covering the block lie
// inside the buffer, five vector loads and a funnel shift per word replace the
// seventeen word loads (one chunk per thread puts every word load of a warp on 32
// different cache lines); otherwise load_block_global.
__device__ __forceinline__ void load_block_units(const uint8_t *base, uint64_t len, uint64_t off, uint32_t m[16]) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(base) + off;
    const uintptr_t buf_lo = reinterpret_cast<uintptr_t>(base);
    const uintptr_t buf_hi = buf_lo + len;
    const uintptr_t a16 = addr & ~static_cast<uintptr_t>(15);
    if (a16 >= buf_lo && a16 + kBlockLen + 16 <= buf_hi) {
        // every word funnel-shifted out of two neighbouring loaded words; the unit
        // offset (r >> 2) is the same for every chunk of an input, so the switch does
        // not diverge
        const uint4 *p = reinterpret_cast<const uint4 *>(a16);
        uint32_t u[20];
#pragma unroll
        for (int k = 0; k < 5; ++k) {
            const uint4 w = __ldg(p + k);
            u[4 * k + 0] = w.x;
            u[4 * k + 1] = w.y;
            u[4 * k + 2] = w.z;
            u[4 * k + 3] = w.w;
        }
        const uint32_t r = static_cast<uint32_t>(addr & 15u);
        const uint32_t sh = (r & 3u) * 8u;
        switch (r >> 2) {
#define B3G_SHIFTED_WORDS(Q)                                                            \
    case Q:                                                                             \
        _Pragma("unroll") for (int i = 0; i < 16; ++i) m[i] = __funnelshift_r(u[i + Q], u[i + Q + 1], sh); \
        return;
            B3G_SHIFTED_WORDS(0)
            B3G_SHIFTED_WORDS(1)
            B3G_SHIFTED_WORDS(2)
            B3G_SHIFTED_WORDS(3)
#undef B3G_SHIFTED_WORDS
        }
    }
    load_block_global(base, len, off, m);
}

// ---------------------------------------------------------------------------------
// CV nodes in shared memory.  Node j occupies 16-byte units 2j and 2j+1; unit k is
// stored at k with its low three bits XORed by bits 3..5 (a 128-byte swizzle), so
// that both "thread j writes node j" and "thread t reads nodes 2t, 2t+1" touch 32
// distinct banks per quarter-warp.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t node_unit_addr(uint32_t base, uint32_t unit) {
    const uint32_t phys = unit ^ ((unit >> 3) & 7u);
    return base + phys * 16u;
}

__device__ __forceinline__ void store_node(uint32_t base, uint32_t j, const uint32_t cv[8]) {
    sts128(node_unit_addr(base, 2 * j), make_uint4(cv[0], cv[1], cv[2], cv[3]));
    sts128(node_unit_addr(base, 2 * j + 1), make_uint4(cv[4], cv[5], cv[6], cv[7]));
}

__device__ __forceinline__ void load_node(uint32_t base, uint32_t j, uint32_t cv[8]) {
    uint4 a = lds128(node_unit_addr(base, 2 * j));
    uint4 b = lds128(node_unit_addr(base, 2 * j + 1));
    cv[0] = a.x; cv[1] = a.y; cv[2] = a.z; cv[3] = a.w;
    cv[4] = b.x; cv[5] = b.y; cv[6] = b.z; cv[7] = b.w;
}

// ---------------------------------------------------------------------------------
// Tree reduction of `cnt` consecutive nodes into one (page section
// "Merkle Tree 归约").  Each level pairs nodes (2j, 2j+1); when a level has an odd
// count its last node moves up unchanged.  Level-order pairing with that
// carry-up builds exactly the tree of the binary decomposition folded right to
// left: after level L the array holds the perfect 2^L subtrees of the aligned
// prefix followed, if the count is not a multiple of 2^L, by the right fold of the
// remainder; pairing the last perfect subtree with that fold is the next step of
// the right-to-left fold.
//
// Levels with more than 32 nodes run in shared memory with the active threads
// packed into whole warps; once 32 nodes or fewer are left, warp 0 holds one node
// per lane and finishes with shuffles, without shared memory or barriers.  ROOT
// goes on the final compression when `root` is set.
// ---------------------------------------------------------------------------------

// Warp-level part: lane j holds node j (j < cnt); on return lane 0 holds the root.
__device__ __forceinline__ void warp_tree(uint32_t x[8], uint32_t cnt, const uint32_t key[8], uint32_t mode_flags,
                                          bool root) {
    const uint32_t lane = threadIdx.x & 31u;
    while (cnt > 1) {
        const uint32_t half = cnt >> 1;
        uint32_t l[8], r[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            l[w] = __shfl_sync(0xffffffffu, x[w], (2 * lane) & 31u);
            r[w] = __shfl_sync(0xffffffffu, x[w], (2 * lane + 1) & 31u);
        }
        if (lane < half) {
            parent(key, mode_flags, l, r, root && cnt == 2, x);
        } else if (lane == half && (cnt & 1u)) {
#pragma unroll
            for (int w = 0; w < 8; ++w) x[w] = l[w];  // node cnt-1 moves up
        }
        cnt = (cnt + 1) >> 1;
    }
}

// Block-level part, over the `nthreads` threads that share named barrier `bar_id`.
// On entry node j (j < cnt) is in `nodes` and a barrier has made the stores
// visible.  On return lane 0 of warp 0 (thread 0) holds the root in out[8]; the
// node buffer may be reused after the call.
__device__ __forceinline__ void block_tree(uint32_t nodes, uint32_t cnt, uint32_t tid, uint32_t nthreads,
                                           uint32_t bar_id, const uint32_t key[8], uint32_t mode_flags,
                                           bool root, uint32_t out[8]) {
    while (cnt > 32) {
        const uint32_t half = cnt >> 1;
        uint32_t res[8];
        bool have = false;
        if (tid < half) {
            uint32_t l[8], r[8];
            load_node(nodes, 2 * tid, l);
            load_node(nodes, 2 * tid + 1, r);
            parent(key, mode_flags, l, r, false, res);
            have = true;
        } else if (tid == half && (cnt & 1u)) {
            load_node(nodes, cnt - 1, res);
            have = true;
        }
        named_bar_sync(bar_id, nthreads);
        if (have) store_node(nodes, tid, res);
        named_bar_sync(bar_id, nthreads);
        cnt = (cnt + 1) >> 1;
    }
    if (tid < 32) {
        if (tid < cnt) load_node(nodes, tid, out);
    }
    named_bar_sync(bar_id, nthreads);  // the node buffer is free again
    if (tid < 32) warp_tree(out, cnt, key, mode_flags, root);
}

}  // namespace b3g

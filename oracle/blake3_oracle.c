/*
 * blake3_oracle.c -- plain, slow, obviously correct CPU oracle for the keyed BLAKE3
 * digest of one buffer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link, load or
 * call this file: only the test suite, the smoke check of the build entry and the
 * CPU-baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA library (blake3_merkle_tree_gb300/csrc), and includes
 * nothing from it.
 *
 * What it computes, and where each step comes from:
 *
 *   Source page: "BLAKE3 GPU 400x faster hashing" (qfminer.top, Pearl mining team).
 *   - section "BLAKE3": input split into 1024-byte chunks, each chunk split into
 *     64-byte blocks; every block goes through a 7-round compression that also takes
 *     a 32-byte chaining value (CV), a flag set, the block length and a per-chunk
 *     counter; the first block of a chunk starts from the key (keyed mode, which the
 *     page always uses), every later block starts from the previous block's output
 *     CV; each chunk yields one 32-byte CV; consecutive CVs are then concatenated
 *     into 64-byte blocks and compressed with different flags until one CV is left;
 *     the tree obeys "left subtree full" (a power-of-two chunk count) and "left
 *     subtree at least as large as its right sibling".
 *   - section "压缩函数" (compression function): CHUNK_START on the first block of a
 *     chunk, CHUNK_END on the last; the key is the initial CV.
 *   - section "Merkle Tree 归约" (Merkle tree reduction): parent nodes use counter 0,
 *     block length 64 and flags KEYED_HASH|PARENT; a non-power-of-two leaf count is
 *     split by its binary decomposition (13 = 8 + 4 + 1) and the perfect pieces are
 *     folded right to left.
 *   - section "Kernel 2 和 3": ROOT is set on the final compression only.
 *   - section "不完整块的处理" (incomplete chunks): the last chunk may be shorter than
 *     1024 bytes, even shorter than one 64-byte block; it is zero padded.
 *
 *   The page names but does not print the round function's constants.  These come
 *   from the published BLAKE3 specification (O'Connor, Aumasson, Neves,
 *   Wilcox-O'Hearn, "BLAKE3: one function, fast everywhere", 2020):
 *     IV (the SHA-256 initial hash value), the G function with rotations 16/12/8/7,
 *     the column/diagonal word assignment of a round, the message permutation
 *     applied between rounds, the flag bits (CHUNK_START=1, CHUNK_END=2, PARENT=4,
 *     ROOT=8, KEYED_HASH=16), the state layout (CV, IV[0..3], counter low/high,
 *     block length, flags) and the output v[i] ^ v[i+8].
 *
 * Pins (tests/test_oracle_pins.py):
 *   - IV: closed form (fractional parts of the square roots of the first 8 primes).
 *   - G, its rotations, the column/diagonal assignment and IV: the same round
 *     function, driven with the BLAKE2s schedule (RFC 7693), reproduces
 *     Python's hashlib.blake2s bit for bit.
 *   - Tree shape: recursive largest-power-of-two split == stack merge on every
 *     length 0..65536; the page's 13 = 8+4+1 example; one-chunk identity; the
 *     digest does not depend on the tile size 2^t.
 *   - PARITY UNPINNED (no known-answer source in this environment): the BLAKE3
 *     message permutation, the flag bit values, the placement of counter / block
 *     length / flags in the state and the number of rounds (7) are taken from the
 *     specification as written and are checked only for internal consistency.
 *     The default (unkeyed) mode shares all of that; what it adds, the IV as the
 *     initial CV, is pinned with the IV; its flag word (no mode bit) is unpinned.
 *
 * Plain C11, scalar, no SIMD, no threads.
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------------ */
/* Specification constants (BLAKE3 spec, section 2.1/2.2).                          */
/* ------------------------------------------------------------------------------ */

static const uint32_t ORACLE_IV[8] = {
    0x6A09E667u, 0xBB67AE85u, 0x3C6EF372u, 0xA54FF53Au,
    0x510E527Fu, 0x9B05688Cu, 0x1F83D9ABu, 0x5BE0CD19u,
};

/* message word i of the next round is word PERM[i] of this round */
static const uint8_t ORACLE_PERM[16] = {2, 6, 3, 10, 7, 0, 4, 13, 1, 11, 12, 5, 9, 14, 15, 8};

enum {
    F_CHUNK_START = 1u << 0,
    F_CHUNK_END = 1u << 1,
    F_PARENT = 1u << 2,
    F_ROOT = 1u << 3,
    F_KEYED_HASH = 1u << 4,
};

#define CHUNK_LEN 1024u
#define BLOCK_LEN 64u
#define ROUNDS 7

/* ------------------------------------------------------------------------------ */
/* Little-endian byte <-> word helpers.                                             */
/* ------------------------------------------------------------------------------ */

static uint32_t le32(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static void put_le32(uint8_t *p, uint32_t w) {
    p[0] = (uint8_t)(w);
    p[1] = (uint8_t)(w >> 8);
    p[2] = (uint8_t)(w >> 16);
    p[3] = (uint8_t)(w >> 24);
}

static void words_from_bytes(const uint8_t *bytes, size_t nwords, uint32_t *words) {
    for (size_t i = 0; i < nwords; i++) words[i] = le32(bytes + 4 * i);
}

static void bytes_from_words(const uint32_t *words, size_t nwords, uint8_t *bytes) {
    for (size_t i = 0; i < nwords; i++) put_le32(bytes + 4 * i, words[i]);
}

/* ------------------------------------------------------------------------------ */
/* The quarter-round G and one full round (columns, then diagonals).               */
/* ------------------------------------------------------------------------------ */

static uint32_t rotr32(uint32_t w, unsigned c) { return (w >> c) | (w << (32u - c)); }

static void g(uint32_t v[16], int a, int b, int c, int d, uint32_t x, uint32_t y) {
    v[a] = v[a] + v[b] + x;
    v[d] = rotr32(v[d] ^ v[a], 16);
    v[c] = v[c] + v[d];
    v[b] = rotr32(v[b] ^ v[c], 12);
    v[a] = v[a] + v[b] + y;
    v[d] = rotr32(v[d] ^ v[a], 8);
    v[c] = v[c] + v[d];
    v[b] = rotr32(v[b] ^ v[c], 7);
}

/* s[] is the message in the order the eight G calls consume it: G number i takes
 * s[2i] and s[2i+1].  Both BLAKE3 and BLAKE2s use this round; they differ only in
 * how s is formed, the state set-up, the round count and the output. */
static void round_fn(uint32_t v[16], const uint32_t s[16]) {
    g(v, 0, 4, 8, 12, s[0], s[1]);
    g(v, 1, 5, 9, 13, s[2], s[3]);
    g(v, 2, 6, 10, 14, s[4], s[5]);
    g(v, 3, 7, 11, 15, s[6], s[7]);
    g(v, 0, 5, 10, 15, s[8], s[9]);
    g(v, 1, 6, 11, 12, s[10], s[11]);
    g(v, 2, 7, 8, 13, s[12], s[13]);
    g(v, 3, 4, 9, 14, s[14], s[15]);
}

/* ------------------------------------------------------------------------------ */
/* BLAKE3 compression: 16-word output (the first 8 words are the new CV).           */
/* ------------------------------------------------------------------------------ */

static void compress_words(const uint32_t cv[8], const uint32_t block[16], uint64_t counter,
                           uint32_t block_len, uint32_t flags, uint32_t out[16]) {
    uint32_t v[16];
    uint32_t m[16];
    uint32_t next[16];
    for (int i = 0; i < 8; i++) v[i] = cv[i];
    for (int i = 0; i < 4; i++) v[8 + i] = ORACLE_IV[i];
    v[12] = (uint32_t)counter;
    v[13] = (uint32_t)(counter >> 32);
    v[14] = block_len;
    v[15] = flags;
    memcpy(m, block, sizeof m);
    for (int r = 0; r < ROUNDS; r++) {
        round_fn(v, m);
        if (r + 1 < ROUNDS) {
            for (int i = 0; i < 16; i++) next[i] = m[ORACLE_PERM[i]];
            memcpy(m, next, sizeof m);
        }
    }
    for (int i = 0; i < 8; i++) {
        out[i] = v[i] ^ v[i + 8];
        out[i + 8] = v[i + 8] ^ cv[i];
    }
}

/* ------------------------------------------------------------------------------ */
/* Leaf: the CV of one chunk (page section "BLAKE3", "压缩函数").                    */
/* ------------------------------------------------------------------------------ */

static void chunk_cv_words(const uint32_t key[8], uint32_t mode, const uint8_t *chunk, size_t chunk_len,
                           uint64_t counter, int is_root, uint32_t out_cv[8]) {
    /* number of blocks: ceil(len/64), and one empty block for an empty chunk */
    size_t nblocks = chunk_len == 0 ? 1 : (chunk_len + BLOCK_LEN - 1) / BLOCK_LEN;
    uint32_t cv[8];
    memcpy(cv, key, sizeof cv);
    for (size_t b = 0; b < nblocks; b++) {
        uint8_t padded[BLOCK_LEN];
        uint32_t m[16];
        uint32_t out[16];
        size_t start = b * BLOCK_LEN;
        size_t take = chunk_len - start < BLOCK_LEN ? chunk_len - start : BLOCK_LEN;
        memset(padded, 0, sizeof padded);
        if (take) memcpy(padded, chunk + start, take);
        words_from_bytes(padded, 16, m);
        uint32_t flags = mode;
        if (b == 0) flags |= F_CHUNK_START;
        if (b + 1 == nblocks) {
            flags |= F_CHUNK_END;
            if (is_root) flags |= F_ROOT;
        }
        compress_words(cv, m, counter, (uint32_t)take, flags, out);
        memcpy(cv, out, sizeof cv);
    }
    memcpy(out_cv, cv, sizeof cv);
}

/* ------------------------------------------------------------------------------ */
/* Parent node (page section "Merkle Tree 归约"): counter 0, length 64,             */
/* KEYED_HASH|PARENT, key as the input CV, left CV || right CV as the message.      */
/* ------------------------------------------------------------------------------ */

static void parent_cv_words(const uint32_t key[8], uint32_t mode, const uint32_t left[8], const uint32_t right[8],
                            int is_root, uint32_t out_cv[8]) {
    uint32_t m[16];
    uint32_t out[16];
    memcpy(m, left, 8 * sizeof(uint32_t));
    memcpy(m + 8, right, 8 * sizeof(uint32_t));
    uint32_t flags = mode | F_PARENT | (is_root ? F_ROOT : 0u);
    compress_words(key, m, 0, BLOCK_LEN, flags, out);
    memcpy(out_cv, out, 8 * sizeof(uint32_t));
}

static uint64_t num_chunks(uint64_t len) {
    return len == 0 ? 1 : (len + CHUNK_LEN - 1) / CHUNK_LEN;
}

static size_t chunk_bytes(uint64_t len, uint64_t i) {
    uint64_t start = i * CHUNK_LEN;
    uint64_t rest = len - start;
    return (size_t)(rest < CHUNK_LEN ? rest : CHUNK_LEN);
}

/* ------------------------------------------------------------------------------ */
/* Tree, form 1: recursive.  The left subtree takes the largest power of two        */
/* strictly below the chunk count (left full, left at least as large as the right). */
/* ------------------------------------------------------------------------------ */

static uint64_t largest_pow2_below(uint64_t n) { /* n >= 2 */
    uint64_t p = 1;
    while (p * 2 < n) p *= 2;
    return p;
}

static void subtree_words(const uint32_t key[8], uint32_t mode, const uint8_t *buf, uint64_t len,
                          uint64_t first_chunk, uint64_t nchunks, uint64_t counter_base,
                          int is_root, uint32_t out_cv[8]) {
    if (nchunks == 1) {
        chunk_cv_words(key, mode, buf + first_chunk * CHUNK_LEN, chunk_bytes(len, first_chunk),
                       counter_base + first_chunk, is_root, out_cv);
        return;
    }
    uint64_t left_n = largest_pow2_below(nchunks);
    uint32_t l[8], r[8];
    subtree_words(key, mode, buf, len, first_chunk, left_n, counter_base, 0, l);
    subtree_words(key, mode, buf, len, first_chunk + left_n, nchunks - left_n, counter_base, 0, r);
    parent_cv_words(key, mode, l, r, is_root, out_cv);
}

/* ------------------------------------------------------------------------------ */
/* Tree, form 2: stack merge.  After the CV of chunk i (not the last one) is pushed, */
/* the count c = i + 1 of finished chunks is scanned from its low bit: every       */
/* trailing zero bit closes one complete subtree, so the two top CVs are merged.   */
/* The stack left at the end is the binary decomposition of the chunk count; it is */
/* folded right to left, and the last parent carries ROOT.                         */
/* ------------------------------------------------------------------------------ */

#define MAX_DEPTH 64

static void stack_merge_words(const uint32_t key[8], uint32_t mode, const uint8_t *buf, uint64_t len,
                              uint32_t out_cv[8]) {
    uint32_t stack[MAX_DEPTH + 1][8];
    int depth = 0;
    uint64_t n = num_chunks(len);
    if (n == 1) {
        chunk_cv_words(key, mode, buf, chunk_bytes(len, 0), 0, 1, out_cv);
        return;
    }
    for (uint64_t i = 0; i + 1 < n; i++) {
        chunk_cv_words(key, mode, buf + i * CHUNK_LEN, CHUNK_LEN, i, 0, stack[depth]);
        depth++;
        uint64_t c = i + 1;
        while ((c & 1) == 0) {
            parent_cv_words(key, mode, stack[depth - 2], stack[depth - 1], 0, stack[depth - 2]);
            depth--;
            c >>= 1;
        }
    }
    /* the last chunk, then the right-to-left fold */
    uint32_t right[8];
    chunk_cv_words(key, mode, buf + (n - 1) * CHUNK_LEN, chunk_bytes(len, n - 1), n - 1, 0, right);
    while (depth > 0) {
        parent_cv_words(key, mode, stack[depth - 1], right, depth == 1, right);
        depth--;
    }
    memcpy(out_cv, right, sizeof right);
}

/* ------------------------------------------------------------------------------ */
/* Extendable output (BLAKE3 specification, section 2.6; the page lists it as      */
/* future work).  The root compression is not evaluated once but kept as its       */
/* inputs (CV, message block, block length, flags); output block i is that        */
/* compression with ROOT and the counter set to i, all 16 output words.           */
/* ------------------------------------------------------------------------------ */

typedef struct {
    uint32_t cv[8];
    uint32_t block[16];
    uint32_t block_len;
    uint32_t flags; /* without ROOT */
} root_inputs;

static void root_of_chunk(const uint32_t key[8], uint32_t mode, const uint8_t *chunk, size_t chunk_len,
                          root_inputs *out) {
    size_t nblocks = chunk_len == 0 ? 1 : (chunk_len + BLOCK_LEN - 1) / BLOCK_LEN;
    uint32_t cv[8];
    memcpy(cv, key, sizeof cv);
    for (size_t b = 0; b < nblocks; b++) {
        uint8_t padded[BLOCK_LEN];
        uint32_t m[16];
        size_t start = b * BLOCK_LEN;
        size_t take = chunk_len - start < BLOCK_LEN ? chunk_len - start : BLOCK_LEN;
        memset(padded, 0, sizeof padded);
        if (take) memcpy(padded, chunk + start, take);
        words_from_bytes(padded, 16, m);
        uint32_t flags = mode | (b == 0 ? F_CHUNK_START : 0u);
        if (b + 1 == nblocks) {
            memcpy(out->cv, cv, sizeof cv);
            memcpy(out->block, m, sizeof m);
            out->block_len = (uint32_t)take;
            out->flags = flags | F_CHUNK_END;
            return;
        }
        uint32_t o[16];
        compress_words(cv, m, 0, (uint32_t)take, flags, o);
        memcpy(cv, o, sizeof cv);
    }
}

/* Root inputs of the whole input: the single chunk's last block, or the top
 * parent whose children are the largest power-of-two left subtree and the rest. */
static void root_inputs_of(const uint32_t key[8], uint32_t mode, const uint8_t *buf, uint64_t len,
                           root_inputs *out) {
    uint64_t n = num_chunks(len);
    if (n == 1) {
        root_of_chunk(key, mode, buf, chunk_bytes(len, 0), out);
        return;
    }
    uint64_t left_n = largest_pow2_below(n);
    uint32_t l[8], r[8];
    subtree_words(key, mode, buf, len, 0, left_n, 0, 0, l);
    subtree_words(key, mode, buf, len, left_n, n - left_n, 0, 0, r);
    memcpy(out->cv, key, 8 * sizeof(uint32_t));
    memcpy(out->block, l, 8 * sizeof(uint32_t));
    memcpy(out->block + 8, r, 8 * sizeof(uint32_t));
    out->block_len = BLOCK_LEN;
    out->flags = mode | F_PARENT;
}

static void xof_words(const uint32_t key[8], uint32_t mode, const uint8_t *buf, uint64_t len, uint8_t *out,
                      uint64_t out_len) {
    root_inputs ri;
    root_inputs_of(key, mode, buf, len, &ri);
    for (uint64_t i = 0; i * 64 < out_len; i++) {
        uint32_t o[16];
        uint8_t blk[64];
        compress_words(ri.cv, ri.block, i, ri.block_len, ri.flags | F_ROOT, o);
        bytes_from_words(o, 16, blk);
        uint64_t take = out_len - i * 64 < 64 ? out_len - i * 64 : 64;
        memcpy(out + i * 64, blk, (size_t)take);
    }
}

/* out_len bytes of extendable output; the first 32 equal oracle_keyed_hash. */
void oracle_keyed_hash_xof(const uint8_t *buf, uint64_t len, const uint8_t key[32], uint8_t *out,
                           uint64_t out_len) {
    uint32_t k[8];
    words_from_bytes(key, 8, k);
    xof_words(k, F_KEYED_HASH, buf, len, out, out_len);
}

/* ------------------------------------------------------------------------------ */
/* The default (unkeyed) mode.  Page section "BLAKE3": the first block of a chunk   */
/* starts from an IV by default, from the user's key in keyed mode.  Following the */
/* specification's hash mode, the default mode starts every chunk and every parent */
/* from the IV and sets no mode flag (keyed mode adds KEYED_HASH to every          */
/* compression); the tree and everything else are the same.                       */
/* ------------------------------------------------------------------------------ */

void oracle_hash(const uint8_t *buf, uint64_t len, uint8_t out[32]) {
    uint32_t cv[8];
    stack_merge_words(ORACLE_IV, 0u, buf, len, cv);
    bytes_from_words(cv, 8, out);
}

void oracle_hash_recursive(const uint8_t *buf, uint64_t len, uint8_t out[32]) {
    uint32_t cv[8];
    subtree_words(ORACLE_IV, 0u, buf, len, 0, num_chunks(len), 0, 1, cv);
    bytes_from_words(cv, 8, out);
}

void oracle_hash_xof(const uint8_t *buf, uint64_t len, uint8_t *out, uint64_t out_len) {
    xof_words(ORACLE_IV, 0u, buf, len, out, out_len);
}

/* ------------------------------------------------------------------------------ */
/* BLAKE2s (RFC 7693) on the same round function: used only to pin G, its          */
/* rotations, the column/diagonal assignment and IV against hashlib.blake2s.       */
/* ------------------------------------------------------------------------------ */

static const uint8_t BLAKE2S_SIGMA[10][16] = {
    {0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15},
    {14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3},
    {11, 8, 12, 0, 5, 2, 15, 13, 10, 14, 3, 6, 7, 1, 9, 4},
    {7, 9, 3, 1, 13, 12, 11, 14, 2, 6, 5, 10, 4, 0, 15, 8},
    {9, 0, 5, 7, 2, 4, 10, 15, 14, 1, 11, 12, 6, 8, 3, 13},
    {2, 12, 6, 10, 0, 11, 8, 3, 4, 13, 7, 5, 15, 14, 1, 9},
    {12, 5, 1, 15, 14, 13, 4, 10, 0, 7, 6, 3, 9, 2, 8, 11},
    {13, 11, 7, 14, 12, 1, 3, 9, 5, 0, 15, 4, 8, 6, 2, 10},
    {6, 15, 14, 9, 11, 3, 0, 8, 12, 2, 13, 7, 1, 4, 10, 5},
    {10, 2, 8, 4, 7, 6, 1, 5, 15, 11, 9, 14, 3, 12, 13, 0},
};

static void blake2s_compress(uint32_t h[8], const uint8_t block[64], uint64_t t, int last) {
    uint32_t m[16], s[16], v[16];
    words_from_bytes(block, 16, m);
    for (int i = 0; i < 8; i++) {
        v[i] = h[i];
        v[i + 8] = ORACLE_IV[i];
    }
    v[12] ^= (uint32_t)t;
    v[13] ^= (uint32_t)(t >> 32);
    if (last) v[14] = ~v[14];
    for (int r = 0; r < 10; r++) {
        for (int i = 0; i < 16; i++) s[i] = m[BLAKE2S_SIGMA[r][i]];
        round_fn(v, s);
    }
    for (int i = 0; i < 8; i++) h[i] ^= v[i] ^ v[i + 8];
}

/* ------------------------------------------------------------------------------ */
/* Exported entry points (ctypes).  Keys and CVs are 32 little-endian bytes.        */
/* ------------------------------------------------------------------------------ */

void oracle_iv(uint32_t out[8]) { memcpy(out, ORACLE_IV, sizeof ORACLE_IV); }

void oracle_msg_permutation(uint8_t out[16]) { memcpy(out, ORACLE_PERM, sizeof ORACLE_PERM); }

/* CHUNK_START, CHUNK_END, PARENT, ROOT, KEYED_HASH */
void oracle_flags(uint32_t out[5]) {
    out[0] = F_CHUNK_START;
    out[1] = F_CHUNK_END;
    out[2] = F_PARENT;
    out[3] = F_ROOT;
    out[4] = F_KEYED_HASH;
}

void oracle_compress(const uint8_t cv[32], const uint8_t block[64], uint64_t counter,
                     uint32_t block_len, uint32_t flags, uint8_t out[64]) {
    uint32_t cvw[8], m[16], o[16];
    words_from_bytes(cv, 8, cvw);
    words_from_bytes(block, 16, m);
    compress_words(cvw, m, counter, block_len, flags, o);
    bytes_from_words(o, 16, out);
}

void oracle_chunk_cv(const uint8_t key[32], const uint8_t *chunk, size_t chunk_len,
                     uint64_t counter, int is_root, uint8_t out[32]) {
    uint32_t k[8], cv[8];
    words_from_bytes(key, 8, k);
    chunk_cv_words(k, F_KEYED_HASH, chunk, chunk_len, counter, is_root, cv);
    bytes_from_words(cv, 8, out);
}

void oracle_parent_cv(const uint8_t key[32], const uint8_t left[32], const uint8_t right[32],
                      int is_root, uint8_t out[32]) {
    uint32_t k[8], l[8], r[8], o[8];
    words_from_bytes(key, 8, k);
    words_from_bytes(left, 8, l);
    words_from_bytes(right, 8, r);
    parent_cv_words(k, F_KEYED_HASH, l, r, is_root, o);
    bytes_from_words(o, 8, out);
}

/* The digest, stack-merge form. */
void oracle_keyed_hash(const uint8_t *buf, uint64_t len, const uint8_t key[32], uint8_t out[32]) {
    uint32_t k[8], cv[8];
    words_from_bytes(key, 8, k);
    stack_merge_words(k, F_KEYED_HASH, buf, len, cv);
    bytes_from_words(cv, 8, out);
}

/* The digest, recursive form. */
void oracle_keyed_hash_recursive(const uint8_t *buf, uint64_t len, const uint8_t key[32],
                                 uint8_t out[32]) {
    uint32_t k[8], cv[8];
    words_from_bytes(key, 8, k);
    subtree_words(k, F_KEYED_HASH, buf, len, 0, num_chunks(len), 0, 1, cv);
    bytes_from_words(cv, 8, out);
}

/* Root CV of the subtree made of the chunks of buf[0..len), whose first chunk has
 * global index chunk_offset (the per-chunk counter starts there).  Recursive form. */
void oracle_subtree_cv(const uint8_t *buf, uint64_t len, uint64_t chunk_offset,
                       const uint8_t key[32], int is_root, uint8_t out[32]) {
    uint32_t k[8], cv[8];
    words_from_bytes(key, 8, k);
    subtree_words(k, F_KEYED_HASH, buf, len, 0, num_chunks(len), chunk_offset, is_root, cv);
    bytes_from_words(cv, 8, out);
}

/* All chunk CVs of buf[0..len) (none with ROOT), 32 bytes each, counters from
 * chunk_offset. */
void oracle_chunk_cvs(const uint8_t *buf, uint64_t len, uint64_t chunk_offset,
                      const uint8_t key[32], uint8_t *out) {
    uint32_t k[8], cv[8];
    words_from_bytes(key, 8, k);
    uint64_t n = num_chunks(len);
    for (uint64_t i = 0; i < n; i++) {
        chunk_cv_words(k, F_KEYED_HASH, buf + i * CHUNK_LEN, chunk_bytes(len, i), chunk_offset + i, 0, cv);
        bytes_from_words(cv, 8, out + 32 * i);
    }
}

/* BLAKE2s-256, unkeyed (RFC 7693), built on round_fn. */
void oracle_blake2s_256(const uint8_t *msg, size_t len, uint8_t out[32]) {
    uint32_t h[8];
    memcpy(h, ORACLE_IV, sizeof h);
    h[0] ^= 0x01010000u ^ 32u; /* depth 1, fanout 1, key length 0, digest length 32 */
    size_t off = 0;
    while (len - off > 64) {
        blake2s_compress(h, msg + off, (uint64_t)(off + 64), 0);
        off += 64;
    }
    uint8_t last[64];
    memset(last, 0, sizeof last);
    if (len - off) memcpy(last, msg + off, len - off);
    blake2s_compress(h, last, (uint64_t)len, 1);
    bytes_from_words(h, 8, out);
}

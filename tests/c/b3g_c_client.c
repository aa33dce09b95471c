/* A plain C11 client of the C ABI (include/blake3_gb300.h): no Python, no torch.
 *
 *   b3g_c_client LEN
 *
 * Generates LEN bytes (byte i = (131 i + 7 (i >> 8) + 3) mod 256) and the key
 * (byte i = 7 i + 1), then prints one line of hex each for: blake3_keyed_hash, the
 * streaming hasher fed in three segments, 100 bytes of extendable output,
 * blake3_keyed_hash_host from pageable host memory, the default-mode digest
 * (blake3_hash) and the device status word.
 * Exit status 0 on success, 1 with a message on stderr otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "blake3_gb300.h"

static int check(b3g_status st, const char *what) {
    if (st == B3G_OK) return 0;
    fprintf(stderr, "%s: %s (%s)\n", what, blake3_strerror(st), blake3_last_cuda_error());
    return 1;
}

static void print_hex(const uint8_t *p, size_t n) {
    for (size_t i = 0; i < n; ++i) printf("%02x", p[i]);
    printf("\n");
}

int main(int argc, char **argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: %s LEN\n", argv[0]);
        return 1;
    }
    const uint64_t len = strtoull(argv[1], NULL, 10);
    uint8_t key[32];
    for (int i = 0; i < 32; ++i) key[i] = (uint8_t)(7 * i + 1);
    uint8_t *host = malloc(len ? len : 1);
    if (!host) return 1;
    for (uint64_t i = 0; i < len; ++i) host[i] = (uint8_t)(131u * i + 7u * (i >> 8) + 3u);

    void *d_in = NULL;
    uint8_t *d_out = NULL;
    if (cudaMalloc(&d_in, len ? len : 1) != cudaSuccess || cudaMalloc((void **)&d_out, 128) != cudaSuccess) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 1;
    }
    if (len && cudaMemcpy(d_in, host, len, cudaMemcpyHostToDevice) != cudaSuccess) return 1;
    uint8_t out[128];

    /* one-shot digest */
    if (check(blake3_keyed_hash(d_in, len, key, d_out, NULL), "blake3_keyed_hash")) return 1;
    if (cudaMemcpy(out, d_out, 32, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
    print_hex(out, 32);

    /* streaming hasher, three segments */
    b3g_hasher *h = NULL;
    if (check(blake3_hasher_new(key, &h), "blake3_hasher_new")) return 1;
    const uint64_t a = len / 3, b = 2 * len / 3;
    const uint8_t *p = (const uint8_t *)d_in;
    if (check(blake3_hasher_update(h, p, a, NULL), "update") || check(blake3_hasher_update(h, p + a, b - a, NULL), "update") ||
        check(blake3_hasher_update(h, p + b, len - b, NULL), "update"))
        return 1;
    if (blake3_hasher_count(h) != len) return 1;
    if (check(blake3_hasher_finalize(h, d_out, 32, NULL), "blake3_hasher_finalize")) return 1;
    if (cudaMemcpy(out, d_out, 32, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
    print_hex(out, 32);
    blake3_hasher_free(h);

    /* extendable output */
    if (check(blake3_keyed_hash_xof(d_in, len, key, d_out, 100, NULL), "blake3_keyed_hash_xof")) return 1;
    if (cudaMemcpy(out, d_out, 100, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
    print_hex(out, 100);

    /* from pageable host memory, library-allocated staging */
    if (check(blake3_keyed_hash_host(host, len, key, out, NULL, 0, NULL), "blake3_keyed_hash_host")) return 1;
    print_hex(out, 32);

    /* default (unkeyed) mode */
    if (check(blake3_hash(d_in, len, d_out, NULL), "blake3_hash")) return 1;
    if (cudaMemcpy(out, d_out, 32, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
    print_hex(out, 32);

    uint32_t status = 0;
    if (check(blake3_device_status(&status), "blake3_device_status")) return 1;
    printf("%u\n", status);
    cudaFree(d_in);
    cudaFree(d_out);
    free(host);
    return 0;
}

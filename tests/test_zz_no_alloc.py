"""blake3_keyed_hash_noalloc: the digest for callers that cannot allocate device memory
at hashing time (their GPU memory is owned by another allocator, they cannot accept the
synchronisation an allocation may cause, or their policy forbids allocating after
start-up).  It keeps its CTA roots in a fixed scratch array inside the library.

Checked through the C ABI against the CPU oracle and against blake3_keyed_hash, call
after call (each call reuses the scratch the one before left behind), over every path
the entry point can take: the empty input, inputs shorter than a chunk and than a CTA
subtree (no scratch used), the small-input subtree sizes, a misaligned view, and an
input of more than 760 CTA subtrees (the tile counter in the scratch, two reduction
levels).
This file is collected last on purpose."""

import ctypes

import pytest
import torch

import oracle
from blake3_merkle_tree_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

MAX_LEN = 16 << 30


def _noalloc(lib, dev, key):
    out = torch.empty(32, dtype=torch.uint8, device="cuda")
    st = lib.blake3_keyed_hash_noalloc(dev.data_ptr() if dev.numel() else None, dev.numel(), key, out.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.blake3_strerror(st)
    return bytes(out.cpu().numpy())


# (length, byte offset of the view): 0, 1 and 1023 bytes fit one CTA subtree; 5 MiB + 3
# takes the small-input subtree size; 9 MiB + 5 at offset 3 is misaligned; 300 MiB + 777
# is 2401 subtrees of 128 chunks (more than one per resident CTA: the tile counter; two
# reduction levels)
CASES = [(0, 0), (1, 0), (1023, 0), (5 * (1 << 20) + 3, 0), (9 * (1 << 20) + 5, 3), (300 * (1 << 20) + 777, 0)]


def test_noalloc_matches_the_oracle_call_after_call():
    build.build()
    lib = binding.library()
    key = workloads.key_bytes(7)
    for n, off in CASES:
        host = workloads.uniform_bytes(n % 1000, n)
        buf = torch.empty(n + off, dtype=torch.uint8, device="cuda")
        buf[off:].copy_(host)
        dev = buf[off:]
        want = oracle.keyed_hash(host, key)
        assert _noalloc(lib, dev, key) == want, (n, off)
        assert bytes(binding.blake3_keyed_hash(dev, key).cpu().numpy()) == want, (n, off)
        assert _noalloc(lib, dev, key) == want, (n, off)  # again, on the scratch the call above left
    assert binding.blake3_device_status() == 0


def _oracle_digest_16_parts(host, key):
    """The oracle's digest of a power-of-two number of chunks, from 16 aligned subtrees
    hashed on 16 host threads (the unchanged oracle functions) and folded: the tree of
    2^k chunks is the perfect tree over those subtrees."""
    from concurrent.futures import ThreadPoolExecutor

    n = host.numel()
    part = n // 16
    assert part % 1024 == 0 and (part // 1024) & (part // 1024 - 1) == 0
    with ThreadPoolExecutor(16) as ex:
        cvs = list(ex.map(lambda i: oracle.subtree_cv(host[i * part:(i + 1) * part], key, i * (part // 1024)),
                          range(16)))
    while len(cvs) > 2:
        cvs = [oracle.parent_cv(key, cvs[i], cvs[i + 1]) for i in range(0, len(cvs), 2)]
    return oracle.parent_cv(key, cvs[0], cvs[1], True)


def test_noalloc_at_the_maximum_length():
    """B3G_NOALLOC_MAX_LEN itself: 16 GiB, 131,072 CTA subtrees of 128 chunks, the most
    roots the scratch holds, with the tile counter at its end; twice in a row, against
    the oracle (16 aligned subtrees on host threads, folded)."""
    build.build()
    lib = binding.library()
    key = workloads.key_bytes(11)
    dev = workloads.uniform_bytes(16, MAX_LEN, device="cuda")
    got = [_noalloc(lib, dev, key) for _ in range(2)]
    host = dev.cpu()
    del dev
    torch.cuda.empty_cache()
    want = _oracle_digest_16_parts(host, key)
    assert got[0] == want and got[1] == want
    assert binding.blake3_device_status() == 0


def test_noalloc_rejects_inputs_over_the_limit():
    build.build()
    lib = binding.library()
    out = torch.empty(32, dtype=torch.uint8, device="cuda")
    fake = ctypes.c_void_p(0x10000)  # rejected before anything is launched
    st = lib.blake3_keyed_hash_noalloc(fake, MAX_LEN + 1, bytes(32), out.data_ptr(), None)
    assert st == 3  # B3G_ERR_WORKSPACE

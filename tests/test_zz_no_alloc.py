"""blake3_keyed_hash_noalloc: the digest for callers that cannot allocate device memory
at hashing time (their GPU memory is owned by another allocator, they cannot accept the
synchronisation an allocation may cause, or their policy forbids allocating after
start-up).  It keeps its CTA roots in a fixed scratch array inside the library.

Checked through the C ABI against blake3_keyed_hash, on two calls in a row with
different inputs (the second call reuses the scratch the first one left behind).
This file is collected last on purpose."""

import ctypes

import pytest
import torch

from blake3_merkle_tree_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

MAX_LEN = 16 << 30


def _noalloc(lib, dev, key):
    out = torch.empty(32, dtype=torch.uint8, device="cuda")
    st = lib.blake3_keyed_hash_noalloc(dev.data_ptr() if dev.numel() else None, dev.numel(), key, out.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.blake3_strerror(st)
    return bytes(out.cpu().numpy())


def test_noalloc_matches_blake3_keyed_hash_twice():
    build.build()
    lib = binding.library()
    key = workloads.key_bytes(7)
    # several tiles and a ragged tail, then a larger input with two reduction levels
    sizes = [5 * (1 << 20) + 3, 300 * (1 << 20) + 777]
    for n in sizes:
        dev = workloads.uniform_bytes(n % 1000, n, device="cuda")
        want = bytes(binding.blake3_keyed_hash(dev, key).cpu().numpy())
        assert _noalloc(lib, dev, key) == want, n
    # a single-tile input does not touch the scratch at all
    small = workloads.uniform_bytes(3, 4000, device="cuda")
    assert _noalloc(lib, small, key) == bytes(binding.blake3_keyed_hash(small, key).cpu().numpy())
    assert binding.blake3_device_status() == 0


def test_noalloc_rejects_inputs_over_the_limit():
    build.build()
    lib = binding.library()
    out = torch.empty(32, dtype=torch.uint8, device="cuda")
    fake = ctypes.c_void_p(0x10000)  # rejected before anything is launched
    st = lib.blake3_keyed_hash_noalloc(fake, MAX_LEN + 1, bytes(32), out.data_ptr(), None)
    assert st == 3  # B3G_ERR_WORKSPACE

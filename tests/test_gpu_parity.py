"""GPU parity: every entry point of the C ABI against the CPU oracle, bit-exact.

Inputs are seeded and synthetic (blake3_merkle_tree_gb300.workloads).  Sizes span
several CTA tiles and a ragged tail; the full-size workloads are in
test_gpu_fullsize.py.
"""

import numpy as np
import pytest
import torch

import oracle
from blake3_merkle_tree_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

KEY = workloads.key_bytes(1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blake3_merkle_tree_gb300 import build

    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.library()
    yield
    assert binding.blake3_device_status() == 0


def _gpu_digest(host: torch.Tensor, key) -> bytes:
    d = host.cuda()
    out = binding.blake3_keyed_hash(d, key)
    return bytes(out.cpu().numpy())


def test_one_mib_config():
    w = workloads.WORKLOADS["1MiB"]
    data = w.data()
    assert _gpu_digest(data, w.key()) == oracle.keyed_hash(data, w.key())


@pytest.mark.parametrize("length", workloads.ragged_lengths())
def test_ragged_sweep(length):
    w = workloads.ragged_workload(length)
    data = w.data()
    assert _gpu_digest(data, w.key()) == oracle.keyed_hash(data, w.key()), length


def test_empty_input_null_pointer():
    out = torch.empty(32, dtype=torch.uint8, device="cuda")
    st = binding.library().blake3_keyed_hash(None, 0, KEY, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert bytes(out.cpu().numpy()) == oracle.keyed_hash(b"", KEY)


@pytest.mark.parametrize("length", [1, 63, 1024, 5000, 256 * 1024 + 3, 700 * 1024 + 100])
@pytest.mark.parametrize("offset", [1, 3, 4, 8, 15])
def test_misaligned_inputs(length, offset):
    host = workloads.uniform_bytes(length + 7, length + offset)
    dev = host.cuda()
    view = dev[offset:]
    got = bytes(binding.blake3_keyed_hash(view, KEY).cpu().numpy())
    assert got == oracle.keyed_hash(host[offset:], KEY)


@pytest.mark.parametrize("length", [0, 1, 1024, 1025, 13 * 1024 + 7, 255 * 1024, 256 * 1024, 257 * 1024 - 1,
                                    600 * 1024 + 9])
@pytest.mark.parametrize("chunk_offset", [0, 5, 1 << 32])
def test_chunk_cvs(length, chunk_offset):
    host = workloads.uniform_bytes(90 + length, length)
    got = binding.blake3_keyed_chunk_cvs(host.cuda(), KEY, chunk_offset).cpu().numpy()
    ref = oracle.chunk_cvs(host, KEY, chunk_offset)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("leaves_log2", [5, 6, 7, 8])
@pytest.mark.parametrize("length", [1024, 31 * 1024 + 1, 64 * 1024, 1000 * 1024 + 1, 2048 * 1024])
def test_tile_roots(leaves_log2, length):
    host = workloads.uniform_bytes(7 + length, length)
    roots = binding.blake3_keyed_tile_roots(host.cuda(), KEY, 0, leaves_log2).cpu().numpy()
    tile = (1 << leaves_log2) * 1024
    ntiles = -(-length // tile)
    assert roots.shape == (ntiles, 32)
    for i in range(ntiles):
        ref = oracle.subtree_cv(host[i * tile:(i + 1) * tile], KEY, i << leaves_log2, is_root=False)
        assert bytes(roots[i]) == ref, i


@pytest.mark.parametrize("leaves_log2", [5, 6, 7, 8])
@pytest.mark.parametrize("group_log2", [1, 2, 3, 5, 10])
@pytest.mark.parametrize("length", [13 * 1024 + 7, 777 * 1024, 5000 * 1024 + 333])
def test_digest_independent_of_tile_and_group_size(leaves_log2, group_log2, length):
    """Page section "Kernel 1": 2^t is free, so the digest must not depend on it."""
    host = workloads.uniform_bytes(length, length)
    ref = oracle.keyed_hash(host, KEY)
    d = host.cuda()
    tiles = binding.blake3_tile_count(length, leaves_log2)
    if tiles == 1:
        roots = binding.blake3_keyed_tile_roots(d, KEY, 0, leaves_log2, is_root=True)
        got = bytes(roots[0].cpu().numpy())
    else:
        roots = binding.blake3_keyed_tile_roots(d, KEY, 0, leaves_log2)
        got = bytes(binding.blake3_keyed_reduce_cvs(roots, KEY, True, group_log2).cpu().numpy())
    assert got == ref


@pytest.mark.parametrize("count", [1, 2, 3, 13, 32, 33, 100, 1024, 1025, 3000])
def test_reduce_cvs_against_oracle_tree(count):
    """Random CVs as leaves: the reduction must build the left-full, left-large tree."""
    cvs = workloads.uniform_bytes(4242 + count, 32 * count).reshape(count, 32)
    leaves = [bytes(cvs[i].numpy()) for i in range(count)]

    def fold(xs, is_root):
        if len(xs) == 1:
            return xs[0]
        p = 1
        while p * 2 < len(xs):
            p *= 2
        return oracle.parent_cv(KEY, fold(xs[:p], False), fold(xs[p:], False), is_root)

    for group_log2 in (1, 4, 10):
        got = bytes(binding.blake3_keyed_reduce_cvs(cvs.cuda(), KEY, count > 1, group_log2).cpu().numpy())
        assert got == fold(leaves, count > 1), (count, group_log2)


@pytest.mark.parametrize("length,chunk_offset", [(1024, 0), (1024, 7), (4 * 1024, 4), (64 * 1024, 64),
                                                 (1024 * 1024, 1 << 20), (300 * 1024 + 5, 512),
                                                 (13 * 1024 + 7, 16)])
@pytest.mark.parametrize("is_root", [False, True])
def test_subtree_root(length, chunk_offset, is_root):
    host = workloads.uniform_bytes(length + 11, length)
    got = bytes(binding.blake3_keyed_subtree_root(host.cuda(), KEY, chunk_offset, is_root).cpu().numpy())
    assert got == oracle.subtree_cv(host, KEY, chunk_offset, is_root)


def test_subtree_roots_compose_to_the_digest():
    """Two 512-chunk halves hashed as subtrees, then one parent with ROOT == the digest."""
    length = 1024 * 1024
    host = workloads.uniform_bytes(31, length)
    d = host.cuda()
    left = binding.blake3_keyed_subtree_root(d[:512 * 1024], KEY, 0)
    right = binding.blake3_keyed_subtree_root(d[512 * 1024:], KEY, 512)
    top = oracle.parent_cv(KEY, bytes(left.cpu().numpy()), bytes(right.cpu().numpy()), True)
    assert top == oracle.keyed_hash(host, KEY)
    with pytest.raises(binding.B3GError):
        binding.blake3_keyed_subtree_root(d[512 * 1024:], KEY, 256)


def test_workspace_variant_and_streams():
    w = workloads.WORKLOADS["1MiB"]
    host = w.data()
    d = host.cuda()
    ref = oracle.keyed_hash(host, w.key())
    ws = torch.empty(binding.blake3_workspace_size(d.numel()), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = binding.blake3_keyed_hash_ws(d, w.key(), ws, stream=s)
    s.synchronize()
    assert bytes(out.cpu().numpy()) == ref
    with pytest.raises(binding.B3GError):
        binding.blake3_keyed_hash_ws(d, w.key(), ws[:16])


def test_bf16_matrix_config():
    w = workloads.WORKLOADS["bf16_256MiB"]
    host = w.data()
    assert _gpu_digest(host, w.key()) == oracle.keyed_hash(host, w.key())


def test_generator_same_bytes_on_gpu_and_cpu():
    for seed, n in ((4, 1 << 20), (6, 3 * (1 << 20) + 777)):
        a = workloads.uniform_bytes(seed, n, device="cuda").cpu()
        b = workloads.uniform_bytes(seed, n)
        assert torch.equal(a, b)


@pytest.mark.parametrize("length", [2 * 1024, 33 * 1024 + 5, 300 * 1024 + 3, (1 << 20), (1 << 20) + 1,
                                    4 * 128 * 1024 * 8 - 7])
def test_fused_final_reduction_option(length):
    """With the fused-final option the last CTA reduces the tile CVs itself."""
    host = workloads.uniform_bytes(length + 9, length)
    d = host.cuda()
    ref = oracle.keyed_hash(host, KEY)
    binding.blake3_set_option(binding.B3G_OPT_FUSED_FINAL, 1)
    try:
        for _ in range(2):  # the ticket must be re-zeroed on every call
            assert bytes(binding.blake3_keyed_hash(d, KEY).cpu().numpy()) == ref
        ws = torch.empty(binding.blake3_workspace_size(length), dtype=torch.uint8, device="cuda")
        ws.fill_(0xAB)  # a dirty workspace
        assert bytes(binding.blake3_keyed_hash_ws(d, KEY, ws).cpu().numpy()) == ref
        assert bytes(binding.blake3_keyed_subtree_root(d, KEY, 0, False).cpu().numpy()) == \
            oracle.subtree_cv(host, KEY, 0, False)
    finally:
        binding.blake3_set_option(binding.B3G_OPT_FUSED_FINAL, 0)


@pytest.mark.parametrize("r", list(range(1, 16)))
def test_every_misalignment_residue(r):
    """Inputs starting at every byte offset mod 16 take the plain-load kernel: its
    16-byte-unit loads with shifts (inner blocks), word loads (blocks near the ends) and
    byte loads (the ragged tail) all give the oracle's digest and chunk CVs."""
    n = 300 * 1024 + 77
    host = workloads.uniform_bytes(900 + r, n + 32)
    d = host.cuda()
    x = d[r:r + n]
    ref = host[r:r + n]
    assert bytes(binding.blake3_keyed_hash(x, KEY).cpu().numpy()) == oracle.keyed_hash(ref, KEY)
    assert bytes(binding.blake3_hash(x).cpu().numpy()) == oracle.hash(ref)
    cvs = binding.blake3_keyed_chunk_cvs(x, KEY).cpu().numpy()
    assert (cvs == oracle.chunk_cvs(ref, KEY)).all()


@pytest.mark.parametrize("offset", [0, 5])
def test_dynamic_tile_schedule_gives_the_static_roots(offset):
    """Tiles taken from a zeroed counter (more tiles than resident CTAs, ragged tail,
    aligned and misaligned) give the same roots as the static order, and those roots are
    the oracle's subtree CVs.  Every tile takes from the counter exactly once, and the
    last take puts it back to zero, so the second call reuses it without a clear."""
    n = 200 * (1 << 20) + 777
    host = workloads.uniform_bytes(31, n)
    buf = torch.empty(n + offset, dtype=torch.uint8, device="cuda")
    buf[offset:].copy_(host)
    dev = buf[offset:]
    tiles = binding.blake3_tile_count(n, -1)
    assert tiles > 760
    static = binding.blake3_keyed_tile_roots(dev, KEY)
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        dyn = binding.blake3_keyed_tile_roots(dev, KEY, tile_counter=counter)
        assert torch.equal(dyn, static)
        # n_tiles takes in all, the last of which resets it (fewer or more leave it non-zero)
        assert int(counter.item()) == 0
    roots = static.cpu().numpy()
    per = 128 * 1024
    for t in (0, 1, 759, 760, 761, tiles - 2, tiles - 1):
        want = oracle.subtree_cv(host[t * per:min(n, (t + 1) * per)], KEY, t * 128)
        assert bytes(roots[t]) == want, t


@pytest.mark.parametrize("tiles,offset", [(761, 0), (4097, 0), (761, 3)])
def test_one_shot_digest_with_tile_counter(tiles, offset):
    """Above 760 tiles the one-shot digest takes tiles from a counter that it zeroes in its
    workspace (761 tiles: two reduction levels, 4097: three).  A dirty workspace, reused
    call after call, gives the oracle's digest, keyed and in the default mode, aligned and
    misaligned."""
    n = tiles * 128 * 1024 - 5000  # a partial last tile and a partial last chunk
    host = workloads.uniform_bytes(tiles, n)
    buf = torch.empty(n + offset, dtype=torch.uint8, device="cuda")
    buf[offset:].copy_(host)
    dev = buf[offset:]
    want = oracle.keyed_hash(host, KEY)
    ws = torch.full((binding.blake3_workspace_size(n),), 0xA5, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        assert bytes(binding.blake3_keyed_hash_ws(dev, KEY, ws).cpu().numpy()) == want
    assert bytes(binding.blake3_keyed_hash(dev, KEY).cpu().numpy()) == want
    if tiles == 761 and offset == 0:
        assert bytes(binding.blake3_hash_ws(dev, ws).cpu().numpy()) == oracle.hash(host)


@pytest.mark.parametrize("length,offset", [(9 << 20, 0), ((10 << 20) - 1, 0), (10 << 20, 0), ((12 << 20) + 5, 3),
                                           ((18 << 20) + 777, 0), ((19 << 20) - 1, 8)])
def test_one_shot_digest_around_the_subtree_size_rule(length, offset):
    """The one-shot digest chooses its CTA subtree size from the length: 32 to 64 chunks
    below 80 subtrees of 128, 128 chunks from 80 of them on (10 MiB) even with fewer than
    one CTA per SM.  Lengths on both sides of that step, aligned and misaligned, against
    the oracle, with the workspace the size function gives."""
    host = workloads.uniform_bytes(length + offset, length)
    buf = torch.empty(length + offset, dtype=torch.uint8, device="cuda")
    buf[offset:].copy_(host)
    dev = buf[offset:]
    want = oracle.keyed_hash(host, KEY)
    ws = torch.full((max(16, binding.blake3_workspace_size(length)),), 0x5A, dtype=torch.uint8, device="cuda")
    assert bytes(binding.blake3_keyed_hash_ws(dev, KEY, ws).cpu().numpy()) == want
    assert bytes(binding.blake3_keyed_hash(dev, KEY).cpu().numpy()) == want

"""GPU parity of the extendable output and of the streaming hasher against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from blake3_merkle_tree_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

KEY = workloads.key_bytes(11)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blake3_merkle_tree_gb300 import build

    build.build()
    binding.library()
    yield
    assert binding.blake3_device_status() == 0


@pytest.mark.parametrize("length", [0, 1, 64, 1024, 1025, 2048, 13 * 1024 + 7, 300 * 1024 + 3, 3 * (1 << 20) + 5])
@pytest.mark.parametrize("out_len", [0, 1, 31, 32, 33, 64, 65, 1000, 4096 + 7])
def test_xof(length, out_len):
    host = workloads.uniform_bytes(length + 3, length)
    got = binding.blake3_keyed_hash_xof(host.cuda(), KEY, out_len)
    ref = oracle.keyed_hash_xof(host, KEY, out_len)
    assert bytes(got.cpu().numpy()) == ref


def test_xof_misaligned_output_and_long_output():
    host = workloads.uniform_bytes(5, (1 << 20) + 17)
    d = host.cuda()
    buf = torch.zeros((8 << 20) + 64, dtype=torch.uint8, device="cuda")
    out = buf[3:3 + (8 << 20) + 5]
    binding.blake3_keyed_hash_xof(d, KEY, out.numel(), out=out)
    ref = oracle.keyed_hash_xof(host, KEY, out.numel())
    assert bytes(out.cpu().numpy()) == ref
    assert int(buf[:3].sum()) == 0 and int(buf[3 + out.numel():].sum()) == 0  # nothing written outside
    assert bytes(out[:32].cpu().numpy()) == bytes(binding.blake3_keyed_hash(d, KEY).cpu().numpy())


def _splits(total, parts, seed):
    rng = np.random.default_rng(seed)
    cuts = sorted(int(x) for x in rng.integers(0, total + 1, parts - 1)) if total and parts > 1 else []
    pts = [0] + cuts + [total]
    return [(pts[i], pts[i + 1]) for i in range(len(pts) - 1)]


@pytest.mark.parametrize("total", [0, 1, 1023, 1024, 1025, 2048, 2049, 5000, 64 * 1024, 300 * 1024 + 3,
                                   (4 << 20) + 777])
@pytest.mark.parametrize("parts", [1, 2, 3, 7, 20])
def test_hasher_random_segments(total, parts):
    host = workloads.uniform_bytes(total + 101, total)
    d = host.cuda()
    h = binding.Hasher(KEY)
    for a, b in _splits(total, parts, seed=total * 31 + parts):
        h.update(d[a:b])
    assert h.count == total
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)
    assert bytes(h.finalize(200).cpu().numpy()) == oracle.keyed_hash_xof(host, KEY, 200)
    h.close()


@pytest.mark.parametrize("seg", [1024, 4096, 256 * 1024, 1 << 20])
def test_hasher_chunk_aligned_segments(seg):
    total = 6 * seg + 1024 * 3
    host = workloads.uniform_bytes(seg, total)
    d = host.cuda()
    h = binding.Hasher(KEY)
    for a in range(0, total, seg):
        h.update(d[a:a + seg])
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)


def test_hasher_finalize_then_continue_and_reset():
    total = 3 * (1 << 20) + 99
    host = workloads.uniform_bytes(77, total)
    d = host.cuda()
    h = binding.Hasher(KEY)
    for cut in (1000, 5000, 70 * 1024, 1 << 20):
        h.update(d[h.count:cut])
        assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host[:cut], KEY), cut
    h.update(d[h.count:])
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)
    h.reset()
    assert h.count == 0
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(b"", KEY)
    h.update(d[:5000])
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host[:5000], KEY)


def test_hasher_large_matches_one_shot():
    """64 MiB segments with a ragged end: equal to the one-shot GPU digest and the oracle."""
    w = workloads.WORKLOADS["bf16_256MiB"]
    host = w.data()
    d = host.cuda()
    h = binding.Hasher(w.key())
    seg = 64 << 20
    for a in range(0, d.numel(), seg - 777):
        h.update(d[a:a + seg - 777])
    got = bytes(h.finalize().cpu().numpy())
    assert got == bytes(binding.blake3_keyed_hash(d, w.key()).cpu().numpy())
    assert got == oracle.keyed_hash(host, w.key())


@pytest.mark.parametrize("length", [0, 1, 1024, 1025, (1 << 20) + 3, (9 << 20) + 777])
@pytest.mark.parametrize("staging_mib", [0, 2, 4])
def test_hash_from_host_memory(length, staging_mib):
    """Host input copied in overlapping segments (pinned and pageable) == the oracle digest."""
    host = workloads.uniform_bytes(length + 5, length)
    pinned = torch.empty(length, dtype=torch.uint8, pin_memory=True)
    pinned.copy_(host)
    staging = None
    if staging_mib:
        staging = torch.empty(3328 + (staging_mib << 20), dtype=torch.uint8, device="cuda")
    ref = oracle.keyed_hash(host, KEY)
    assert binding.blake3_keyed_hash_host(pinned, KEY, staging) == ref
    assert binding.blake3_keyed_hash_host(host, KEY, staging) == ref


def test_hash_from_host_rejects_small_staging():
    host = torch.zeros(5000, dtype=torch.uint8)
    staging = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.B3GError):
        binding.blake3_keyed_hash_host(host, KEY, staging)


def test_hasher_very_large_piece():
    """A piece of more than 1024 CTA subtrees inside one update (chunks 2^18 .. 2^19):
    the multi-level reduction branch of the batched push."""
    total = 2048 + (600 << 20) + 5
    host = workloads.uniform_bytes(600, total)
    d = host.cuda()
    h = binding.Hasher(KEY)
    h.update(d[:2048])
    h.update(d[2048:])
    got = bytes(h.finalize().cpu().numpy())
    assert got == bytes(binding.blake3_keyed_hash(d, KEY).cpu().numpy())
    assert got == oracle.keyed_hash(host, KEY)


def test_hasher_many_small_segments():
    """About 140 MiB in segments of 1 B .. 3 MB: they collect in the 64 MiB accumulation
    buffer, which is pushed twice; digests taken in between push the buffered chunks
    onto a copy of the stack only."""
    total = (140 << 20) + 12345
    host = workloads.uniform_bytes(1400, total)
    d = host.cuda()
    rng = np.random.default_rng(1400)
    h = binding.Hasher(KEY)
    checks = {30 << 20, 90 << 20}
    a = 0
    while a < total:
        n = int(min(total - a, rng.integers(1, 3_000_000)))
        if rng.random() < 0.1:
            n = int(min(total - a, rng.integers(1, 2048)))
        h.update(d[a:a + n])
        a += n
        hit = [c for c in checks if c <= a]
        for c in hit:
            checks.discard(c)
            got = bytes(h.finalize().cpu().numpy())
            assert got == bytes(binding.blake3_keyed_hash(d[:a], KEY).cpu().numpy()), a
    assert h.count == total
    got = bytes(h.finalize().cpu().numpy())
    assert got == oracle.keyed_hash(host, KEY)
    assert bytes(h.finalize(100).cpu().numpy()) == oracle.keyed_hash_xof(host, KEY, 100)


def test_hasher_buffer_growth_and_mixed_sizes():
    """Small, larger-than-buffer and exactly-buffer-sized segments in turn; every prefix
    digest equals the one-shot digest of that prefix."""
    sizes = [5, 3000, (70 << 20) + 13, 1 << 20, 64 << 20, 100, 1024, 2047, (64 << 20) - 1, 1, 9 << 20]
    total = sum(sizes)
    host = workloads.uniform_bytes(1401, total)
    d = host.cuda()
    h = binding.Hasher(KEY)
    a = 0
    for n in sizes:
        h.update(d[a:a + n])
        a += n
        got = bytes(h.finalize().cpu().numpy())
        assert got == bytes(binding.blake3_keyed_hash(d[:a], KEY).cpu().numpy()), (n, a)
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)
    h.reset()
    h.update(d[:500])
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host[:500], KEY)
    h.update(d[500:2048])
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host[:2048], KEY)


@pytest.mark.parametrize("sizes", [[4096, 8192], [1024, 1024], [2048], [1024, 1], [1, 1023, 1024, 1024],
                                   [5000, 1 << 20, 3 << 20]])
def test_hasher_finalize_buffered_whole_chunks(sizes):
    """The buffer holds only whole chunks (or one chunk and a byte) at finalize."""
    total = sum(sizes)
    host = workloads.uniform_bytes(1402 + total, total)
    d = host.cuda()
    h = binding.Hasher(KEY)
    a = 0
    for n in sizes:
        h.update(d[a:a + n])
        a += n
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)
    assert bytes(h.finalize(96).cpu().numpy()) == oracle.keyed_hash_xof(host, KEY, 96)


def test_hasher_updates_captured_in_a_cuda_graph():
    """Updates captured into a CUDA graph and replayed once give the oracle digest: under
    capture the side stream rejoins the capturing stream completely and the buffer does not
    grow (no allocation outside the stream)."""
    total = 3 * 1024 + (5 << 20) + 333
    host = workloads.uniform_bytes(1500, total)
    d = host.cuda()
    binding.blake3_keyed_hash(d, KEY)  # first-use set-up (status word, occupancy) outside the capture
    h = binding.Hasher(KEY)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    cuts = [0, 700, 3 * 1024 + 5, (2 << 20) + 77, total]
    with torch.cuda.graph(g, stream=s):
        for a, b in zip(cuts[:-1], cuts[1:]):
            h.update(d[a:b])
    g.replay()
    torch.cuda.synchronize()
    assert h.count == total
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_hasher_update_many_matches_oracle(seed):
    """Many device segments in one call (including empty ones, misaligned starts and a
    few that do not fit the buffer) == the oracle digest of their concatenation."""
    rng = np.random.default_rng(4000 + seed)
    sizes = [int(x) for x in rng.integers(0, 3000, 300)]
    sizes[10] = 0
    sizes[50] = (2 << 20) + 3
    if seed == 1:
        sizes[100] = (70 << 20) + 5  # larger than the accumulation buffer
    if seed == 2:
        sizes = [int(x) for x in rng.integers(1, 700, 1500)]  # more than one launch's worth
    if seed == 3:  # two full 1024-segment launches, then a 128-segment one
        sizes = [int(x) for x in rng.integers(1, 400, 2100)]
    total = sum(sizes)
    host = workloads.uniform_bytes(4100 + seed, total + 64)
    d = host.cuda()
    segs, a = [], 0
    for n in sizes:  # consecutive slices of one buffer: segments start at any byte
        segs.append((a, n))
        a += n
    tensors = [d[x:x + n] for x, n in segs]
    h = binding.Hasher(KEY)
    h.update_many(tensors[:7]).update_many(tensors[7:])
    assert h.count == total
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host[:total], KEY)
    g = binding.Hasher()
    g.update_many(tensors)
    assert bytes(g.finalize().cpu().numpy()) == oracle.hash(host[:total])


def test_hasher_update_many_equals_separate_updates():
    host = workloads.uniform_bytes(4200, 5 << 20)
    d = host.cuda()
    cuts = [0, 1, 1025, 4096, 70000, 70001, 1 << 20, (3 << 20) + 7, 5 << 20]
    tensors = [d[x:y] for x, y in zip(cuts[:-1], cuts[1:])]
    one = binding.Hasher(KEY)
    for t in tensors:
        one.update(t)
    many = binding.Hasher(KEY).update_many(tensors)
    assert bytes(one.finalize().cpu().numpy()) == bytes(many.finalize().cpu().numpy())
    assert bytes(many.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)


@pytest.mark.parametrize("cut", [0, 700, 1024, 1025, 5000, (3 << 20) + 11, (70 << 20) + 3])
@pytest.mark.parametrize("keyed", [True, False])
def test_hasher_checkpoint_and_resume(cut, keyed):
    """Export after `cut` bytes, resume in a new hasher (the old one freed), finish: the
    digest and extendable output equal the oracle's for the whole input."""
    total = cut + (2 << 20) + 333
    host = workloads.uniform_bytes(7000 + cut, total)
    d = host.cuda()
    h = binding.Hasher(KEY if keyed else None)
    for a in range(0, cut, 1 << 20):
        h.update(d[a:min(cut, a + (1 << 20))])
    state = h.export()
    assert len(state) == binding.library().blake3_hasher_export_size(h._h)
    before = bytes(h.finalize().cpu().numpy())
    h.close()
    r = binding.Hasher.from_state(state)
    assert r.count == cut
    assert bytes(r.finalize().cpu().numpy()) == before
    r.update(d[cut:cut + 5]).update(d[cut + 5:])
    ref = oracle.keyed_hash(host, KEY) if keyed else oracle.hash(host)
    assert bytes(r.finalize().cpu().numpy()) == ref
    xof = oracle.keyed_hash_xof(host, KEY, 96) if keyed else oracle.hash_xof(host, 96)
    assert bytes(r.finalize(96).cpu().numpy()) == xof
    assert r.export() != state  # the state moved on


@pytest.fixture
def unbatched():
    binding.blake3_set_option(binding.B3G_OPT_STREAM_UNBATCHED, 1)
    yield
    binding.blake3_set_option(binding.B3G_OPT_STREAM_UNBATCHED, 0)


@pytest.mark.parametrize("keyed", [True, False])
def test_hasher_unbatched_path(unbatched, keyed):
    """The one-piece-at-a-time push (a subtree launch and a merge launch per piece, the
    path beyond the batch limits) gives the oracle digest on ragged and large segments."""
    total = 3 * 1024 + (70 << 20) + (5 << 20) + 777
    host = workloads.uniform_bytes(7100 + keyed, total)
    d = host.cuda()
    cuts = [0, 2048, 3 * 1024 + 5, (70 << 20) + 11, (72 << 20) + 1, total]
    h = binding.Hasher(KEY if keyed else None)
    for a, b in zip(cuts[:-1], cuts[1:]):
        h.update(d[a:b])
    ref = oracle.keyed_hash(host, KEY) if keyed else oracle.hash(host)
    assert bytes(h.finalize().cpu().numpy()) == ref
    rng = np.random.default_rng(7101)
    sizes = [int(x) for x in rng.integers(1, 5000, 200)]
    segs, a = [], 0
    for n in sizes:
        segs.append(d[a:a + n])
        a += n
    g = binding.Hasher(KEY if keyed else None)
    g.update_many(segs)
    g.update(d[a:])
    assert bytes(g.finalize().cpu().numpy()) == ref

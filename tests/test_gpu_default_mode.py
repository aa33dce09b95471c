"""GPU parity of the default (unkeyed) mode against the oracle: one-shot digests on the
ragged length set, misaligned inputs, caller workspace, extendable output, the streaming
hasher, host input, and a large input."""

import numpy as np
import pytest
import torch

import oracle
from blake3_merkle_tree_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blake3_merkle_tree_gb300 import build

    build.build()
    binding.library()
    yield
    assert binding.blake3_device_status() == 0


@pytest.mark.parametrize("length", workloads.ragged_lengths()[:13] + workloads.ragged_lengths()[13:29])
def test_default_mode_digest(length):
    host = workloads.uniform_bytes(length, length)
    d = host.cuda()
    got = bytes(binding.blake3_hash(d).cpu().numpy())
    assert got == oracle.hash(host)
    # the mode matters: the keyed digest under the IV bytes differs
    iv = b"".join(w.to_bytes(4, "little") for w in oracle.iv())
    assert got != bytes(binding.blake3_keyed_hash(d, iv).cpu().numpy())


@pytest.mark.parametrize("offset", [1, 3, 8])
@pytest.mark.parametrize("length", [1025, 64 * 1024 + 1, (1 << 20) + 9])
def test_default_mode_misaligned(offset, length):
    host = workloads.uniform_bytes(length + offset, length + offset)
    d = host.cuda()[offset:]
    assert bytes(binding.blake3_hash(d).cpu().numpy()) == oracle.hash(host[offset:])


@pytest.mark.parametrize("length", [0, 5000, 300 * 1024 + 17, (9 << 20) + 777])
def test_default_mode_workspace(length):
    host = workloads.uniform_bytes(length + 11, length)
    d = host.cuda()
    ws = torch.empty(max(16, binding.blake3_workspace_size(length)), dtype=torch.uint8, device="cuda")
    assert bytes(binding.blake3_hash_ws(d, ws).cpu().numpy()) == oracle.hash(host)


@pytest.mark.parametrize("length", [0, 1, 1024, 1025, 13 * 1024 + 7, 3 * (1 << 20) + 5])
@pytest.mark.parametrize("out_len", [0, 31, 32, 65, 4096 + 7])
def test_default_mode_xof(length, out_len):
    host = workloads.uniform_bytes(length + 13, length)
    got = binding.blake3_hash_xof(host.cuda(), out_len)
    assert bytes(got.cpu().numpy()) == oracle.hash_xof(host, out_len)


@pytest.mark.parametrize("total", [0, 1023, 1025, 70 * 1024 + 3, (5 << 20) + 77])
def test_default_mode_hasher(total):
    host = workloads.uniform_bytes(total + 17, total)
    d = host.cuda()
    rng = np.random.default_rng(total)
    cuts = sorted(int(x) for x in rng.integers(0, total + 1, 6)) if total else []
    pts = [0] + cuts + [total]
    h = binding.Hasher()
    for a, b in zip(pts[:-1], pts[1:]):
        h.update(d[a:b])
    assert bytes(h.finalize().cpu().numpy()) == oracle.hash(host)
    assert bytes(h.finalize(100).cpu().numpy()) == oracle.hash_xof(host, 100)
    h.close()


@pytest.mark.parametrize("length", [0, 1025, (3 << 20) + 5])
def test_default_mode_from_host(length):
    host = workloads.uniform_bytes(length + 19, length)
    assert binding.blake3_hash_host(host) == oracle.hash(host)


def test_default_mode_large():
    """256 MiB + 777 B (2^18 chunks and a tail): many CTA subtrees, two reduction levels."""
    n = (256 << 20) + 777
    host = workloads.uniform_bytes(2024, n)
    d = host.cuda()
    got = bytes(binding.blake3_hash(d).cpu().numpy())
    assert got == oracle.hash(host)
    h = binding.Hasher()
    h.update(d[:(100 << 20) + 3]).update(d[(100 << 20) + 3:])
    assert bytes(h.finalize().cpu().numpy()) == got

"""GPU parity at the full workload sizes, in the launch configuration the benchmark
times: the whole digest against the CPU oracle, plus sampled chunk CVs and sampled
CTA subtree roots that the oracle computes one by one."""

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


@pytest.mark.parametrize("name", ["4GiB", "12GiB+777"])
def test_full_size_digest_and_samples(name):
    w = workloads.WORKLOADS[name]
    key = w.key()
    dev = w.data(device="cuda")
    got = bytes(binding.blake3_keyed_hash(dev, key).cpu().numpy())

    n = dev.numel()
    nchunks = -(-n // 1024)
    rng = np.random.default_rng(n)
    # sampled chunk CVs (first, last = the partial one for the ragged size, random)
    cvs = binding.blake3_keyed_chunk_cvs(dev, key)
    idx = sorted(set([0, nchunks - 1, nchunks // 2] + list(rng.integers(0, nchunks, 64))))
    # sampled CTA subtree roots (the default subtree size)
    per_tile = 1 << binding.library().blake3_default_leaves_log2()
    roots = binding.blake3_keyed_tile_roots(dev, key)
    ntiles = roots.shape[0]
    tidx = sorted(set([0, ntiles - 1] + list(rng.integers(0, ntiles, 8))))
    cvs_h = cvs.cpu().numpy()
    roots_h = roots.cpu().numpy()
    del cvs, roots
    host = dev.cpu()
    del dev
    torch.cuda.empty_cache()
    for i in idx:
        i = int(i)
        chunk = host[i * 1024:(i + 1) * 1024]
        assert bytes(cvs_h[i]) == oracle.chunk_cv(key, chunk, i), i
    for t in tidx:
        t = int(t)
        part = host[t * per_tile * 1024:(t + 1) * per_tile * 1024]
        assert bytes(roots_h[t]) == oracle.subtree_cv(part, key, t * per_tile), t
    assert got == oracle.keyed_hash(host, key)

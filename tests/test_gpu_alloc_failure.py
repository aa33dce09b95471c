"""Failure handling without a GPU fault: the library's allocation hook
(B3G_OPT_FAIL_ALLOC) makes one device allocation fail as if the device were out of
memory.  The call that needed it returns B3G_ERR_CUDA, the context stays usable, and
the next call gives the oracle's digest; the streaming hasher's optional buffer
degrades to the small one."""

import pytest
import torch

import oracle
from blake3_merkle_tree_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

KEY = workloads.key_bytes(61)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from blake3_merkle_tree_gb300 import build

    build.build()
    binding.library()
    yield
    binding.blake3_set_option(binding.B3G_OPT_FAIL_ALLOC, 0)
    assert binding.blake3_device_status() == 0


def _fail_next(n=1):
    binding.blake3_set_option(binding.B3G_OPT_FAIL_ALLOC, n)


def test_one_shot_workspace_failure_then_recovery():
    host = workloads.uniform_bytes(6100, (8 << 20) + 5)
    d = host.cuda()
    _fail_next()
    with pytest.raises(binding.B3GError) as err:
        binding.blake3_keyed_hash(d, KEY)
    assert err.value.status == 4 and "out of memory" in str(err.value)
    assert bytes(binding.blake3_keyed_hash(d, KEY).cpu().numpy()) == oracle.keyed_hash(host, KEY)
    # the hook counts allocations: the second one fails, the first goes through
    _fail_next(2)
    assert bytes(binding.blake3_hash(d).cpu().numpy()) == oracle.hash(host)
    with pytest.raises(binding.B3GError):
        binding.blake3_hash(d)
    assert bytes(binding.blake3_hash(d).cpu().numpy()) == oracle.hash(host)


def test_xof_and_host_input_failures():
    host = workloads.uniform_bytes(6101, (3 << 20) + 7)
    d = host.cuda()
    _fail_next()
    with pytest.raises(binding.B3GError):
        binding.blake3_keyed_hash_xof(d, KEY, 100)
    assert bytes(binding.blake3_keyed_hash_xof(d, KEY, 100).cpu().numpy()) == oracle.keyed_hash_xof(host, KEY, 100)
    _fail_next()
    with pytest.raises(binding.B3GError):
        binding.blake3_keyed_hash_host(host, KEY)  # its own staging allocation fails
    assert binding.blake3_keyed_hash_host(host, KEY) == oracle.keyed_hash(host, KEY)


def test_hasher_buffer_growth_failure_degrades_gracefully():
    """The 64 MiB buffer cannot be had: the hasher keeps its 1 KiB buffer, same digest."""
    total = (6 << 20) + 333
    host = workloads.uniform_bytes(6102, total)
    d = host.cuda()
    h = binding.Hasher(KEY)
    h.update(d[:100])
    _fail_next()  # the growth on the next small update
    for a in range(100, total, 300_000):
        h.update(d[a:a + 300_000])
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)


def test_hasher_push_failure_then_reset():
    total = (70 << 20) + 9  # the second segment exceeds the 64 MiB buffer: it must push
    host = workloads.uniform_bytes(6103, total)
    d = host.cuda()
    h = binding.Hasher(KEY)
    h.update(d[:5000])
    _fail_next()  # the scratch of the push of the next (large) segment
    with pytest.raises(binding.B3GError):
        h.update(d[5000:])
    h.reset()
    h.update(d[:5000]).update(d[5000:])
    assert bytes(h.finalize().cpu().numpy()) == oracle.keyed_hash(host, KEY)
    _fail_next()
    with pytest.raises(binding.B3GError):
        binding.Hasher(KEY)  # its state allocation fails
    torch.cuda.synchronize()

"""The bounded device-side wait gives up, reports it, and leaves the context usable.

Uses a probe kernel that waits on a barrier nothing completes (no fault, no trap,
no endless loop): the same wait routine guards every barrier wait of the hashing
kernels."""

import pytest
import torch

import oracle
from blake3_merkle_tree_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_survives():
    from blake3_merkle_tree_gb300 import build

    build.build()
    assert binding.blake3_selftest_bounded_wait(200_000) is True
    key = workloads.key_bytes(1)
    host = workloads.uniform_bytes(5, 300 * 1024 + 1)
    got = bytes(binding.blake3_keyed_hash(host.cuda(), key).cpu().numpy())
    assert got == oracle.keyed_hash(host, key)
    assert binding.blake3_device_status() == 0


def test_per_call_status_word_in_stream_order():
    """A caller's status word tells one call's outcome from a copy on the caller's stream,
    without synchronising the device: the probe's given-up wait sets the bit there (and
    not in the per-device word); a hash through blake3_keyed_hash_ex on the same stream
    leaves a zeroed word clear and gives the oracle's digest."""
    from blake3_merkle_tree_gb300 import build

    build.build()
    s = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    seen = torch.zeros(1, dtype=torch.int32).pin_memory()
    key = workloads.key_bytes(1)
    host = workloads.uniform_bytes(7, 3 * 128 * 1024 + 77)
    data = host.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        binding.blake3_selftest_bounded_wait_ex(50_000, status, stream=s)
        seen.copy_(status, non_blocking=True)
    s.synchronize()
    assert int(seen.item()) == binding.B3G_DEVICE_STATUS_TIMEOUT
    with torch.cuda.stream(s):
        status.zero_()
        out = binding.blake3_keyed_hash_ex(data, key, status, stream=s)
        ws = torch.empty(max(16, binding.blake3_workspace_size(data.numel())), dtype=torch.uint8, device="cuda")
        out_ws = binding.blake3_keyed_hash_ex(data, key, status, workspace=ws, stream=s)
        seen.copy_(status, non_blocking=True)
    s.synchronize()
    assert int(seen.item()) == 0
    ref = oracle.keyed_hash(host, key)
    assert bytes(out.cpu().numpy()) == ref and bytes(out_ws.cpu().numpy()) == ref
    assert binding.blake3_device_status() == 0

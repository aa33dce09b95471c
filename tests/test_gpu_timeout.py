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

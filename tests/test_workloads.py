"""The seeded input generators: torch (any device) == numpy == scalar restatement."""

import numpy as np
import pytest
import torch

from blake3_merkle_tree_gb300 import workloads


def test_torch_numpy_scalar_agree():
    for seed in (0, 1, 6, 1000):
        words = workloads.splitmix_words_scalar(seed, 0, 40)
        ref = b"".join(w.to_bytes(8, "little") for w in words)
        t = workloads.uniform_bytes(seed, 317, slice_bytes=64).numpy().tobytes()
        n = workloads.numpy_uniform_bytes(seed, 317).tobytes()
        assert t == ref[:317] == n


def test_slices_are_position_independent():
    full = workloads.uniform_bytes(6, 4096).numpy()
    again = workloads.uniform_bytes(6, 4096, slice_bytes=1000).numpy()
    assert np.array_equal(full, again)


def test_keys_and_lengths():
    assert len(workloads.key_bytes(1)) == 32
    assert workloads.key_bytes(1) != workloads.key_bytes(3)
    lens = workloads.ragged_lengths()
    assert len(lens) == 77 and lens[:3] == [0, 1, 63]
    assert all(1 <= n <= 4 << 20 for n in lens[13:])


def test_workload_sizes():
    w = workloads.WORKLOADS
    assert w["1MiB"].nbytes == 1 << 20
    assert w["4GiB"].nbytes == 1 << 32
    assert w["12GiB+777"].nbytes == 12_884_902_665
    assert w["bf16_256MiB"].nbytes == 268_435_456
    small = workloads.bf16_matrix_bytes(2, rows=4, cols=8)
    assert small.dtype == torch.uint8 and small.numel() == 64


def test_byte_ranges_of_a_stream_match_its_prefix():
    """A slice [start, start + n) made on its own (start a multiple of 8) equals the same
    bytes of the whole stream: what every rank of a sharded digest generates."""
    import torch

    w = workloads.WORKLOADS["12GiB+777"]
    whole = workloads.uniform_bytes(w.data_seed, 3 << 20)
    for start, n in [(0, 1000), (8, 4096), (128 * 1024, 777), ((1 << 20) + 16, 1 << 20)]:
        assert torch.equal(w.data_range(start, n), whole[start:start + n])
    with pytest.raises(ValueError):
        workloads.uniform_bytes(6, 16, start=4)
    with pytest.raises(ValueError):
        workloads.WORKLOADS["bf16_256MiB"].data_range(0, 16)

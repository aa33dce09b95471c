"""The compression-only self-test kernel: it runs, and it leaves its sink alone."""
import pytest
import torch

from blake3_merkle_tree_gb300 import binding

pytestmark = pytest.mark.gpu


def test_compress_rate_kernel_runs_without_touching_memory():
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    binding.blake3_selftest_compress_rate(props.multi_processor_count, 8, sink)
    binding.blake3_selftest_compress_rate(1, 1, sink[1:])
    torch.cuda.synchronize()
    assert sink.tolist() == [0, 0, 0, 0]
    with pytest.raises(binding.B3GError):
        binding.blake3_selftest_compress_rate(0, 1, sink)

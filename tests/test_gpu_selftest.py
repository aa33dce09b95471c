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


def _oracle_chain(key: bytes, g: int, chain: int) -> bytes:
    import oracle

    block = b"".join((((16 * g + i) * 0x9E3779B9) & 0xFFFFFFFF).to_bytes(4, "little") for i in range(16))
    cv = key
    for j in range(chain):
        cv = oracle.compress(cv, block, j, 64, oracle.flags()["KEYED_HASH"])[:32]
    return cv


@pytest.mark.parametrize("lanes", [1, 4])
@pytest.mark.parametrize("chain", [1, 16])
def test_compression_with_several_lanes_per_chunk_matches_the_oracle(lanes, chain):
    """The latency self-test's chains (one lane per chain, and four lanes per chain with
    the state split by columns) give the oracle's chained compressions."""
    from blake3_merkle_tree_gb300 import workloads

    key = workloads.key_bytes(11)
    n = 32 // lanes
    cvs = torch.zeros((n, 32), dtype=torch.uint8, device="cuda")
    cycles = torch.zeros(1, dtype=torch.int64, device="cuda")
    binding.blake3_selftest_compress_latency(lanes, chain, key, cvs, cycles)
    torch.cuda.synchronize()
    got = cvs.cpu().numpy()
    for g in range(n):
        assert bytes(got[g]) == _oracle_chain(key, g, chain), (lanes, chain, g)
    assert int(cycles.item()) > 0

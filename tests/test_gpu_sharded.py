"""The sharded digest on the GPU.

Several ranks cannot run on one GPU, so the per-rank work is emulated rank by rank on
the same device: each rank's slice goes through `blake3_keyed_tile_roots` with its own
chunk offset, and the roots, in rank order, are folded by `blake3_keyed_reduce_cvs`.
The result must equal the one-shot digest and, for small sizes, the oracle's. A
one-rank NCCL group then runs the real `ShardedDigest` (leaf launch, all-gather, fold),
from device memory and from pinned host memory.
"""

import os
import socket

import pytest
import torch

import oracle
from blake3_merkle_tree_gb300 import binding, sharded, workloads

pytestmark = pytest.mark.gpu

KEY = workloads.key_bytes(7)
TILE = sharded.TILE_BYTES


def _emulated(whole: torch.Tensor, world: int) -> bytes:
    n = whole.numel()
    t = sharded.tile_count(n)
    roots = []
    for r in range(world):
        t0, t1 = sharded.shard_tiles(n, world, r)
        start, end = sharded.shard_range(n, world, r)
        if t1 == t0:
            assert start == end
            continue
        out = torch.empty((t1 - t0, 32), dtype=torch.uint8, device="cuda")
        binding.blake3_keyed_tile_roots(whole[start:end], KEY, t0 * sharded.TILE_CHUNKS, sharded.TILE_LOG2,
                                        t == 1, out)
        roots.append(out)
    cvs = torch.cat(roots)
    assert cvs.shape[0] == t
    if t == 1:
        return bytes(cvs[0].cpu().numpy())
    return bytes(binding.blake3_keyed_reduce_cvs(cvs, KEY, True).cpu().numpy())


@pytest.mark.parametrize("world", [2, 3, 5, 8])
@pytest.mark.parametrize("n", [0, 1, 1024, TILE, TILE + 1, 3 * TILE - 1, 13 * TILE + 777])
def test_emulated_ranks_match_oracle(world, n):
    host = workloads.uniform_bytes(6, n)
    got = _emulated(host.cuda(), world)
    assert got == oracle.keyed_hash(bytes(host.numpy()), KEY)


@pytest.mark.parametrize("world", [2, 7, 8])
def test_emulated_ranks_match_one_shot_digest_at_scale(world):
    n = (256 << 20) + 777
    d = workloads.uniform_bytes(6, n, device="cuda")
    assert _emulated(d, world) == bytes(binding.blake3_keyed_hash(d, KEY).cpu().numpy())


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture
def one_rank_nccl():
    import torch.distributed as dist

    store = dist.TCPStore("127.0.0.1", _free_port(), 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        yield
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n", [0, 5000, TILE, (64 << 20) + 777])
def test_sharded_digest_in_a_one_rank_group(one_rank_nccl, n):
    d = workloads.uniform_bytes(6, n, device="cuda")
    want = bytes(binding.blake3_keyed_hash(d, KEY).cpu().numpy())
    sd = sharded.ShardedDigest(n, KEY)
    assert (sd.start, sd.end) == (0, n)
    marks = []
    assert bytes(sd(d, after_leaf=lambda: marks.append(1)).cpu().numpy()) == want
    assert marks == [1]
    assert bytes(sd(d).cpu().numpy()) == want  # buffers reused
    host = d.cpu().pin_memory()
    assert bytes(sd.from_host(host, piece_bytes=4 * TILE).cpu().numpy()) == want
    assert bytes(sd.from_host(host).cpu().numpy()) == want
    with pytest.raises(ValueError):
        sd(d[:n - 1] if n else workloads.uniform_bytes(6, 1, device="cuda"))

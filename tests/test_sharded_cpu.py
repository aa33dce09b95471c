"""The sharded digest's host logic on the CPU: gloo ranks, each holding its slice.

The per-tile subtree roots and the fold are computed here by the oracle (test
infrastructure); what is under test is the plan (which tiles and bytes each rank holds),
the gather in rank order and the placement of ROOT. Every rank's digest must equal the
oracle's digest of the whole buffer.
"""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TILE = 128 * 1024
LENGTHS = [0, 1000, TILE, TILE + 1, 3 * TILE, 5 * TILE + 777, 7 * TILE - 5]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_fold(cvs, key, root):
    """Left-full fold of subtree CVs (split at the largest power of two below the count)."""
    import oracle

    if len(cvs) == 1:
        return cvs[0]
    split = 1
    while split * 2 < len(cvs):
        split *= 2
    left = _oracle_fold(cvs[:split], key, False)
    right = _oracle_fold(cvs[split:], key, False)
    return oracle.parent_cv(key, left, right, is_root=root)


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import oracle
    from blake3_merkle_tree_gb300 import sharded, workloads

    def tile_roots(data, key, chunk_offset, is_root, out):
        raw = bytes(data.numpy())
        for j in range(out.shape[0]):
            piece = raw[j * sharded.TILE_BYTES:(j + 1) * sharded.TILE_BYTES]
            cv = oracle.subtree_cv(piece, key, chunk_offset + j * sharded.TILE_CHUNKS, is_root)
            out[j].copy_(torch.frombuffer(bytearray(cv), dtype=torch.uint8))

    def fold(cvs, key, out, workspace):
        leaves = [bytes(cvs[i].numpy()) for i in range(cvs.shape[0])]
        out.copy_(torch.frombuffer(bytearray(_oracle_fold(leaves, key, True)), dtype=torch.uint8))

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        key = workloads.key_bytes(7)
        results = []
        for n in LENGTHS:
            whole = workloads.uniform_bytes(6, n)
            sd = sharded.ShardedDigest(n, key, device="cpu", tile_roots=tile_roots, fold=fold)
            local = whole[sd.start:sd.end]
            digest = bytes(sd(local).numpy())
            results.append((n, sd.start, sd.end, sd.t0, sd.t1, digest))
        q.put((rank, results))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_digest_equals_whole_buffer_digest(world):
    import torch.multiprocessing as mp

    sys.path.insert(0, ROOT)
    import oracle
    from blake3_merkle_tree_gb300 import sharded, workloads

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        results = dict(q.get(timeout=300) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0] * world
    key = workloads.key_bytes(7)
    for i, n in enumerate(LENGTHS):
        expected = oracle.keyed_hash(bytes(workloads.uniform_bytes(6, n).numpy()), key)
        spans = []
        for r in range(world):
            n_r, start, end, t0, t1, digest = results[r][i]
            assert n_r == n
            assert digest == expected, (n, world, r)
            spans.append((start, end, t0, t1))
        # the slices tile the buffer in rank order, on 128-chunk boundaries
        assert spans[0][0] == 0 and spans[-1][1] == n
        for (s0, e0, a0, b0), (s1, e1, a1, b1) in zip(spans, spans[1:]):
            assert e0 == s1 and b0 == a1
        for start, end, t0, t1 in spans:
            assert start == min(t0 * sharded.TILE_BYTES, n)
        # tiles dealt out evenly: the counts differ by at most one
        counts = [t1 - t0 for _, _, t0, t1 in spans]
        assert max(counts) - min(counts) <= 1 and sum(counts) == sharded.tile_count(n)


def test_shard_plan_arithmetic():
    sys.path.insert(0, ROOT)
    from blake3_merkle_tree_gb300 import sharded

    gib12 = 12 * (1 << 30)
    # eight ranks of one 8 x 12 GiB + 777 buffer: 98,304 tiles each, the last one more
    total = 8 * gib12 + 777
    assert sharded.tile_count(total) == 8 * 98304 + 1
    for r in range(8):
        start, end = sharded.shard_range(total, 8, r)
        assert start == r * gib12
        assert end == ((r + 1) * gib12 if r < 7 else total)
    assert sharded.tile_count(0) == 1 and sharded.shard_range(0, 4, 0) == (0, 0)
    assert sharded.shard_range(0, 4, 3) == (0, 0)

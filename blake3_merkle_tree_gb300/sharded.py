"""Keyed BLAKE3 digest of one buffer sharded over the ranks of a process group.

Each rank (one GPU) holds a contiguous slice of the buffer. Every slice starts on a
128-chunk subtree boundary, and every slice but the last also ends on one. The tiles of
128 chunks are dealt out evenly in rank order: rank r takes tiles
[r*T//world, (r+1)*T//world) of the T tiles.

A rank turns its slice into the roots of its tiles with the leaf kernel
(`blake3_keyed_tile_roots`). The chunk counters start at the slice's first chunk, and
no ROOT is set. The roots of all ranks, in rank order, are the left-to-right leaves of
the tree's upper levels; `blake3_keyed_reduce_cvs` folds them and sets ROOT on the
final compression. The same structure appears on the page "BLAKE3 GPU 400x faster
hashing", section "Kernel 2 和 3": the subtree roots of the CTAs are reduced by later
kernels. Every tile is an aligned power-of-two subtree, except possibly the last.
The digest is therefore identical to the digest of the whole buffer on one GPU.

The only exchange is one all-gather of 32 bytes per tile.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

TILE_LOG2 = 7
TILE_CHUNKS = 1 << TILE_LOG2
CHUNK_BYTES = 1024
TILE_BYTES = TILE_CHUNKS * CHUNK_BYTES


def tile_count(total_len: int) -> int:
    """Tiles of 128 chunks in a buffer of `total_len` bytes (an empty buffer is one chunk)."""
    chunks = max(1, -(-total_len // CHUNK_BYTES))
    return -(-chunks // TILE_CHUNKS)


def shard_tiles(total_len: int, world: int, rank: int) -> tuple[int, int]:
    """The tiles [t0, t1) of `rank`."""
    t = tile_count(total_len)
    return rank * t // world, (rank + 1) * t // world


def shard_range(total_len: int, world: int, rank: int) -> tuple[int, int]:
    """The bytes [start, end) that `rank` holds."""
    t0, t1 = shard_tiles(total_len, world, rank)
    return min(t0 * TILE_BYTES, total_len), min(t1 * TILE_BYTES, total_len)


_counters = {}


def _device_tile_roots(data, key, chunk_offset, is_root, out):
    """The rank's tile roots, the tiles taken from a counter zeroed on the current
    stream (dynamic scheduling: the CTAs that run faster take more tiles)."""
    from . import binding

    dev = out.device
    if dev not in _counters:
        _counters[dev] = torch.zeros(4, dtype=torch.int32, device=dev)
    counter = _counters[dev]
    counter.zero_()
    return binding.blake3_keyed_tile_roots(data, key, chunk_offset, TILE_LOG2, is_root, out, tile_counter=counter)


def _device_fold(cvs, key, out, workspace):
    from . import binding

    return binding.blake3_keyed_reduce_cvs(cvs, key, True, -1, out, workspace)


class ShardedDigest:
    """Plans and buffers of a sharded digest of `total_len` bytes over `group`.

    The buffers are allocated once, so that repeated digests allocate nothing.
    `tile_roots(data, key, chunk_offset, is_root, out)` and
    `fold(cvs, key, out, workspace)` default to the CUDA library; the host logic
    (the plan, the gather and the order) does not depend on them.
    """

    def __init__(self, total_len: int, key, group=None, device=None, tile_roots=None, fold=None):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.total_len = total_len
        self.key = bytes(key)
        self.tiles = tile_count(total_len)
        self.t0, self.t1 = shard_tiles(total_len, self.world, self.rank)
        self.start, self.end = shard_range(total_len, self.world, self.rank)
        self.counts = [shard_tiles(total_len, self.world, r)[1] - shard_tiles(total_len, self.world, r)[0]
                       for r in range(self.world)]
        self.per = max(self.counts)
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.tile_roots = tile_roots or _device_tile_roots
        self.fold = fold or _device_fold
        self.local_roots = torch.zeros((self.per, 32), dtype=torch.uint8, device=dev)
        self.gathered = torch.empty((self.world * self.per, 32), dtype=torch.uint8, device=dev)
        self.parts = list(self.gathered.view(self.world, self.per, 32).unbind(0))
        even = all(c == self.per for c in self.counts)
        self.rows = self.gathered if even else torch.empty((self.tiles, 32), dtype=torch.uint8, device=dev)
        self.out = torch.empty(32, dtype=torch.uint8, device=dev)
        self.workspace = None
        if fold is None and self.tiles > 1:
            from . import binding

            need = binding.blake3_reduce_workspace_size(self.tiles)
            self.workspace = torch.empty(max(16, need), dtype=torch.uint8, device=dev)

    def local_bytes(self) -> int:
        return self.end - self.start

    def _check_len(self, nbytes: int) -> None:
        if nbytes != self.end - self.start:
            raise ValueError(f"rank {self.rank} holds bytes [{self.start}, {self.end}): "
                             f"{self.end - self.start} bytes, got {nbytes}")

    def __call__(self, local: torch.Tensor, after_leaf=None) -> torch.Tensor:
        """The digest of the whole buffer, given this rank's slice on its device (the 32
        bytes on every rank).  `after_leaf()`, if given, runs right after the leaf launch."""
        self._check_len(local.numel() * local.element_size())
        n = self.t1 - self.t0
        if n:
            # a buffer of one tile: that tile's root is the digest (ROOT on its last compression)
            self.tile_roots(local, self.key, self.t0 * TILE_CHUNKS, self.tiles == 1, self.local_roots[:n])
        if after_leaf is not None:
            after_leaf()
        return self._finish()

    def from_host(self, host: torch.Tensor, piece_bytes: int = 256 << 20) -> torch.Tensor:
        """The same digest with this rank's slice in (pinned) host memory: the slice is
        copied in tile-aligned pieces on a copy stream, two device slots in turn, and each
        piece's tile roots are computed on the current stream as soon as it has landed."""
        self._check_len(host.numel() * host.element_size())
        piece_bytes -= piece_bytes % TILE_BYTES
        if piece_bytes <= 0:
            raise ValueError("piece_bytes must hold at least one tile")
        total = self.end - self.start
        if not hasattr(self, "_slots") or self._slots[0].numel() < min(piece_bytes, max(total, 1)):
            size = min(piece_bytes, max(total, 1))
            self._slots = [torch.empty(size, dtype=torch.uint8, device=self.device) for _ in range(2)]
            self._copy_stream = torch.cuda.Stream(device=self.device)
        cur = torch.cuda.current_stream(self.device)
        cs = self._copy_stream
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        consumed = [torch.cuda.Event(), torch.cuda.Event()]
        cs.wait_stream(cur)  # the slots are free from here on
        src = host.view(torch.uint8).reshape(-1)
        for i, pos in enumerate(range(0, total, piece_bytes)):
            b = i & 1
            m = min(piece_bytes, total - pos)
            if i >= 2:
                cs.wait_event(consumed[b])
            with torch.cuda.stream(cs):
                self._slots[b][:m].copy_(src[pos:pos + m], non_blocking=True)
                copied[b].record(cs)
            cur.wait_event(copied[b])
            j0 = pos // TILE_BYTES
            j1 = j0 + -(-m // TILE_BYTES)
            self.tile_roots(self._slots[b][:m], self.key, (self.t0 + j0) * TILE_CHUNKS, self.tiles == 1,
                            self.local_roots[j0:j1])
            consumed[b].record(cur)
        if total == 0 and self.t1 > self.t0:  # the empty buffer: one empty tile
            self.tile_roots(self._slots[0][:0], self.key, 0, True, self.local_roots[:1])
        return self._finish()

    def _finish(self) -> torch.Tensor:
        dist.all_gather(self.parts, self.local_roots, group=self.group)
        if self.tiles == 1:  # the one rank that holds the tile computed the digest
            owner = self.counts.index(1)
            self.out.copy_(self.parts[owner][0])
            return self.out
        if self.rows is not self.gathered:
            pos = 0
            for r, c in enumerate(self.counts):
                self.rows[pos:pos + c].copy_(self.parts[r][:c])
                pos += c
        self.fold(self.rows, self.key, self.out, self.workspace)
        return self.out


def sharded_keyed_hash(local: torch.Tensor, total_len: int, key, group=None) -> torch.Tensor:
    """One sharded digest (plans and allocates on every call; see ShardedDigest)."""
    return ShardedDigest(total_len, key, group, device=local.device)(local)

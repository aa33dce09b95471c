"""Seeded synthetic inputs for the keyed BLAKE3 workloads.

This module only makes input bytes and keys; it holds no hashing arithmetic.
The CUDA path and the CPU oracle both take their inputs from here.

Uniform bytes come from a counter-based generator, SplitMix64 (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014, with the
64-bit finaliser used by java.util.SplittableRandom): word ``i`` of stream
``seed`` is ``mix(base(seed) + (i + 1) * GAMMA)``, with
``base(seed) = mix((seed + 1) * GAMMA)``, and each 64-bit word gives 8 bytes in
little-endian order.  Being counter based, any slice of a stream can be made on
any device, and the CPU and the GPU make identical bytes (checked by a test
against a scalar Python restatement).

Workloads (sizes and seeds):
  1 MiB      1,048,576 uniform bytes, data seed 0, key seed 1
  ragged     13 fixed lengths + 64 lengths drawn from stream 1000 in [1, 4 MiB];
             the bytes of length L use seed L; key seed 1
  bf16       256 MiB: a row-major 8192 x 16384 bf16 matrix of N(0, 1) values
             (torch CPU generator seeded with 2, float32 rounded to bf16), key seed 3
  4 GiB      2^32 uniform bytes, data seed 4, key seed 5
  12 GiB+777 12,884,902,665 uniform bytes, data seed 6, key seed 7
  1 GiB      2^30 uniform bytes, data seed 8, key seed 9 (profiling case only)
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1


def _to_i64(x: int) -> int:
    x &= MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


def _mix_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_base(seed: int) -> int:
    return _mix_int((seed + 1) * GAMMA)


def splitmix_words_scalar(seed: int, start: int, count: int) -> list[int]:
    """Plain-Python restatement of the generator (small counts; used by tests)."""
    base = stream_base(seed)
    return [_mix_int(base + (i + 1) * GAMMA) for i in range(start, start + count)]


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    # logical right shift of int64 lanes holding uint64 bit patterns
    return torch.bitwise_and(torch.bitwise_right_shift(z, k), (1 << (64 - k)) - 1)


def _splitmix_words_torch(seed: int, start: int, count: int, device) -> torch.Tensor:
    base = _to_i64(stream_base(seed))
    idx = torch.arange(start + 1, start + 1 + count, dtype=torch.int64, device=device)
    # int64 arithmetic wraps modulo 2^64 on both CPU and CUDA
    z = idx * _to_i64(GAMMA) + base
    z = torch.bitwise_xor(z, _lsr(z, 30)) * _to_i64(MIX1)
    z = torch.bitwise_xor(z, _lsr(z, 27)) * _to_i64(MIX2)
    z = torch.bitwise_xor(z, _lsr(z, 31))
    return z


def uniform_bytes(seed: int, nbytes: int, device="cpu", out: torch.Tensor | None = None,
                  slice_bytes: int = 1 << 28, start: int = 0) -> torch.Tensor:
    """``nbytes`` uniform bytes of stream ``seed``, from byte ``start`` on (a multiple of
    8), as a uint8 tensor on ``device``.

    Made slice by slice (``slice_bytes`` at a time) to bound the temporaries.
    If ``out`` is given it must be a contiguous uint8 tensor of ``nbytes`` elements.
    """
    if start % 8:
        raise ValueError("start must be a multiple of 8")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=device)
    assert out.numel() == nbytes and out.dtype == torch.uint8 and out.is_contiguous()
    slice_bytes = max(8, slice_bytes - slice_bytes % 8)
    pos = 0
    while pos < nbytes:
        take = min(slice_bytes, nbytes - pos)
        nwords = (take + 7) // 8
        words = _splitmix_words_torch(seed, (start + pos) // 8, nwords, out.device)
        # int64 -> little-endian bytes (both CPU and GB300 are little-endian)
        out[pos:pos + take].copy_(words.view(torch.uint8)[:take])
        pos += take
    return out


def key_bytes(seed: int) -> bytes:
    """A 32-byte key: the first 32 bytes of stream ``seed``."""
    words = splitmix_words_scalar(seed, 0, 4)
    return b"".join(w.to_bytes(8, "little") for w in words)


def ragged_lengths() -> list[int]:
    """The ragged-length sweep: 13 fixed lengths and 64 seeded lengths in [1, 4 MiB]."""
    fixed = [0, 1, 63, 64, 65, 1023, 1024, 1025, 2048, 13 * 1024, 13 * 1024 + 7,
             (1 << 20) - 1, (1 << 20) + 1]
    rnd = [1 + (w % (4 << 20)) for w in splitmix_words_scalar(1000, 0, 64)]
    return fixed + rnd


def bf16_matrix_bytes(seed: int = 2, rows: int = 8192, cols: int = 16384) -> torch.Tensor:
    """Bytes of a row-major rows x cols bf16 matrix of N(0,1) values (CPU)."""
    g = torch.Generator().manual_seed(seed)
    m = torch.randn(rows, cols, dtype=torch.float32, generator=g).to(torch.bfloat16)
    return m.contiguous().view(torch.uint8).reshape(-1)


@dataclass(frozen=True)
class Workload:
    name: str
    nbytes: int
    data_seed: int
    key_seed: int
    kind: str = "uniform"  # or "bf16"

    def key(self) -> bytes:
        return key_bytes(self.key_seed)

    def data(self, device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
        if self.kind == "bf16":
            b = bf16_matrix_bytes(self.data_seed)
            assert b.numel() == self.nbytes
            if out is not None:
                out.copy_(b)
                return out
            return b.to(device)
        return uniform_bytes(self.data_seed, self.nbytes, device=device, out=out)

    def data_range(self, start: int, nbytes: int, device="cpu") -> torch.Tensor:
        """Bytes [start, start + nbytes) of this workload's stream, which continues past
        ``self.nbytes`` (a larger buffer of the same kind); uniform workloads only."""
        if self.kind != "uniform":
            raise ValueError("byte ranges are defined for uniform workloads only")
        return uniform_bytes(self.data_seed, nbytes, device=device, start=start)


WORKLOADS = {
    "1MiB": Workload("1MiB", 1 << 20, 0, 1),
    "bf16_256MiB": Workload("bf16_256MiB", 8192 * 16384 * 2, 2, 3, kind="bf16"),
    "4GiB": Workload("4GiB", 1 << 32, 4, 5),
    "12GiB+777": Workload("12GiB+777", 12 * (1 << 30) + 777, 6, 7),
    # profiling case: larger than L2, small enough for a many-pass profiler capture
    "1GiB": Workload("1GiB", 1 << 30, 8, 9),
}

RAGGED_KEY_SEED = 1


def ragged_workload(length: int) -> Workload:
    return Workload(f"ragged_{length}", length, length, RAGGED_KEY_SEED)


def numpy_uniform_bytes(seed: int, nbytes: int) -> np.ndarray:
    """Independent numpy restatement of ``uniform_bytes`` (uint64 arithmetic)."""
    nwords = (nbytes + 7) // 8
    idx = np.arange(1, nwords + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = idx * np.uint64(GAMMA) + np.uint64(stream_base(seed))
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
        z = z ^ (z >> np.uint64(31))
    return z.astype("<u8").view(np.uint8)[:nbytes]

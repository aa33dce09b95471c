"""CPU oracle for the keyed BLAKE3 digest (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and the
two share no code: this wrapper loads ``liboracle.so`` built from
``blake3_oracle.c`` (plain scalar C11) and only marshals arguments.

The computation and its citations are in ``blake3_oracle.c``.  Parity of the
BLAKE3 message permutation, flag values, state layout and round count is
unpinned in this environment (no known-answer source); see that file's header.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "blake3_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CHUNK_LEN = 1024
BLOCK_LEN = 64
OUT_LEN = 32


def build(force: bool = False) -> str:
    """Compile liboracle.so with the host C compiler (no CUDA involved)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        c_u8p = ctypes.c_void_p
        u64 = ctypes.c_uint64
        lib.oracle_iv.argtypes = [ctypes.c_void_p]
        lib.oracle_msg_permutation.argtypes = [ctypes.c_void_p]
        lib.oracle_flags.argtypes = [ctypes.c_void_p]
        lib.oracle_compress.argtypes = [c_u8p, c_u8p, u64, ctypes.c_uint32, ctypes.c_uint32, c_u8p]
        lib.oracle_chunk_cv.argtypes = [c_u8p, c_u8p, ctypes.c_size_t, u64, ctypes.c_int, c_u8p]
        lib.oracle_parent_cv.argtypes = [c_u8p, c_u8p, c_u8p, ctypes.c_int, c_u8p]
        lib.oracle_keyed_hash.argtypes = [c_u8p, u64, c_u8p, c_u8p]
        lib.oracle_keyed_hash_recursive.argtypes = [c_u8p, u64, c_u8p, c_u8p]
        lib.oracle_subtree_cv.argtypes = [c_u8p, u64, u64, c_u8p, ctypes.c_int, c_u8p]
        lib.oracle_chunk_cvs.argtypes = [c_u8p, u64, u64, c_u8p, c_u8p]
        lib.oracle_blake2s_256.argtypes = [c_u8p, ctypes.c_size_t, c_u8p]
        lib.oracle_keyed_hash_xof.argtypes = [c_u8p, u64, c_u8p, c_u8p, u64]
        lib.oracle_hash.argtypes = [c_u8p, u64, c_u8p]
        lib.oracle_hash_recursive.argtypes = [c_u8p, u64, c_u8p]
        lib.oracle_hash_xof.argtypes = [c_u8p, u64, c_u8p, u64]
        for name in ("oracle_iv", "oracle_msg_permutation", "oracle_flags", "oracle_compress",
                     "oracle_chunk_cv", "oracle_parent_cv", "oracle_keyed_hash",
                     "oracle_keyed_hash_recursive", "oracle_subtree_cv", "oracle_chunk_cvs",
                     "oracle_blake2s_256", "oracle_keyed_hash_xof", "oracle_hash", "oracle_hash_recursive",
                     "oracle_hash_xof"):
            getattr(lib, name).restype = None
        _lib = lib
        return lib


def _buf(data):
    """(pointer, length, keepalive) for bytes, bytearray, numpy array or CPU tensor."""
    if data is None:
        return None, 0, None
    if isinstance(data, (bytes, bytearray, memoryview)):
        arr = np.frombuffer(bytes(data), dtype=np.uint8)
    elif isinstance(data, np.ndarray):
        arr = np.ascontiguousarray(data).view(np.uint8).reshape(-1)
    else:  # torch tensor on the CPU
        t = data.contiguous()
        if t.device.type != "cpu":
            raise ValueError("oracle inputs must live in host memory")
        arr = t.view(-1).numpy().view(np.uint8).reshape(-1)
    if arr.size == 0:
        return None, 0, arr
    return arr.ctypes.data, arr.size, arr


def _key(key) -> bytes:
    key = bytes(key)
    if len(key) != 32:
        raise ValueError("key must be 32 bytes")
    return key


def iv() -> list[int]:
    out = (ctypes.c_uint32 * 8)()
    _load().oracle_iv(out)
    return list(out)


def msg_permutation() -> list[int]:
    out = (ctypes.c_uint8 * 16)()
    _load().oracle_msg_permutation(out)
    return list(out)


def flags() -> dict[str, int]:
    out = (ctypes.c_uint32 * 5)()
    _load().oracle_flags(out)
    return dict(zip(("CHUNK_START", "CHUNK_END", "PARENT", "ROOT", "KEYED_HASH"), out))


def compress(cv: bytes, block: bytes, counter: int, block_len: int, flags_: int) -> bytes:
    """Full 64-byte compression output; the first 32 bytes are the new CV."""
    if len(cv) != 32 or len(block) != 64:
        raise ValueError("cv must be 32 bytes and block 64 bytes")
    out = ctypes.create_string_buffer(64)
    _load().oracle_compress(bytes(cv), bytes(block), counter, block_len, flags_, out)
    return out.raw


def chunk_cv(key, chunk, counter: int, is_root: bool = False) -> bytes:
    p, n, keep = _buf(chunk)
    if n > CHUNK_LEN:
        raise ValueError("a chunk holds at most 1024 bytes")
    out = ctypes.create_string_buffer(32)
    _load().oracle_chunk_cv(_key(key), p, n, counter, int(is_root), out)
    del keep
    return out.raw


def parent_cv(key, left: bytes, right: bytes, is_root: bool = False) -> bytes:
    out = ctypes.create_string_buffer(32)
    _load().oracle_parent_cv(_key(key), bytes(left), bytes(right), int(is_root), out)
    return out.raw


def keyed_hash(data, key) -> bytes:
    """The 32-byte keyed digest (stack-merge tree)."""
    p, n, keep = _buf(data)
    out = ctypes.create_string_buffer(32)
    _load().oracle_keyed_hash(p, n, _key(key), out)
    del keep
    return out.raw


def keyed_hash_recursive(data, key) -> bytes:
    """The 32-byte keyed digest (recursive largest-power-of-two split)."""
    p, n, keep = _buf(data)
    out = ctypes.create_string_buffer(32)
    _load().oracle_keyed_hash_recursive(p, n, _key(key), out)
    del keep
    return out.raw


def subtree_cv(data, key, chunk_offset: int = 0, is_root: bool = False) -> bytes:
    p, n, keep = _buf(data)
    out = ctypes.create_string_buffer(32)
    _load().oracle_subtree_cv(p, n, chunk_offset, _key(key), int(is_root), out)
    del keep
    return out.raw


def chunk_cvs(data, key, chunk_offset: int = 0) -> np.ndarray:
    """All chunk CVs, as a (n_chunks, 32) uint8 array, none with ROOT."""
    p, n, keep = _buf(data)
    nchunks = max(1, -(-n // CHUNK_LEN))
    out = np.zeros((nchunks, 32), dtype=np.uint8)
    _load().oracle_chunk_cvs(p, n, chunk_offset, _key(key), out.ctypes.data)
    del keep
    return out


def keyed_hash_xof(data, key, out_len: int) -> bytes:
    """out_len bytes of extendable output (root compression repeated with counter i)."""
    p, n, keep = _buf(data)
    out = ctypes.create_string_buffer(max(1, out_len))
    _load().oracle_keyed_hash_xof(p, n, _key(key), out, out_len)
    del keep
    return out.raw[:out_len]


def hash(data) -> bytes:  # noqa: A001 - the mode's name
    """The 32-byte digest in the default (unkeyed) mode: the IV is the initial CV and no
    compression carries KEYED_HASH (stack-merge tree)."""
    p, n, keep = _buf(data)
    out = ctypes.create_string_buffer(32)
    _load().oracle_hash(p, n, out)
    del keep
    return out.raw


def hash_recursive(data) -> bytes:
    """The default-mode digest, recursive tree form."""
    p, n, keep = _buf(data)
    out = ctypes.create_string_buffer(32)
    _load().oracle_hash_recursive(p, n, out)
    del keep
    return out.raw


def hash_xof(data, out_len: int) -> bytes:
    """out_len bytes of default-mode extendable output."""
    p, n, keep = _buf(data)
    out = ctypes.create_string_buffer(max(1, out_len))
    _load().oracle_hash_xof(p, n, out, out_len)
    del keep
    return out.raw[:out_len]


def blake2s_256(data) -> bytes:
    p, n, keep = _buf(data)
    out = ctypes.create_string_buffer(32)
    _load().oracle_blake2s_256(p, n, out)
    del keep
    return out.raw

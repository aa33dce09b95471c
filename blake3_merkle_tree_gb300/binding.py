"""ctypes binding of libb3g.so: the C ABI of include/blake3_gb300.h, same names.

Argument marshalling only (torch tensors -> device pointers and byte counts, key
bytes, the current CUDA stream); every step of the computation runs in the CUDA
library.  There is no fallback: if the library is missing or a call fails, the
call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libb3g.so")

B3G_OK = 0
B3G_DEVICE_STATUS_TIMEOUT = 1
STATUS_NAMES = {0: "B3G_OK", 1: "B3G_ERR_NULL", 2: "B3G_ERR_ALIGN", 3: "B3G_ERR_WORKSPACE",
                4: "B3G_ERR_CUDA", 5: "B3G_ERR_TIMEOUT", 6: "B3G_ERR_ARG"}

_lock = threading.Lock()
_lib = None


class B3GError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def library() -> ctypes.CDLL:
    """Load libb3g.so (it must have been built, e.g. by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libb3g.so not built at {LIB_PATH}; run blake3_merkle_tree_gb300.build")
        lib = ctypes.CDLL(LIB_PATH)
        vp, u64, i32, sz = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t
        sigs = {
            "blake3_strerror": (ctypes.c_char_p, [i32]),
            "blake3_last_cuda_error": (ctypes.c_char_p, []),
            "blake3_default_leaves_log2": (i32, []),
            "blake3_kernel_config": (ctypes.c_char_p, []),
            "blake3_set_option": (i32, [i32, ctypes.c_int64]),
            "blake3_keyed_hash": (i32, [vp, u64, vp, vp, vp]),
            "blake3_workspace_size": (sz, [u64]),
            "blake3_keyed_hash_ws": (i32, [vp, u64, vp, vp, vp, sz, vp]),
            "blake3_keyed_hash_noalloc": (i32, [vp, u64, vp, vp, vp]),
            "blake3_keyed_hash_ex": (i32, [vp, u64, vp, vp, vp, sz, vp, vp]),
            "blake3_selftest_bounded_wait_ex": (i32, [ctypes.c_uint32, vp, vp]),
            "blake3_selftest_compress_latency": (i32, [i32, ctypes.c_uint32, vp, vp, vp, vp]),
            "blake3_keyed_chunk_cvs": (i32, [vp, u64, u64, vp, vp, vp]),
            "blake3_keyed_subtree_root": (i32, [vp, u64, u64, vp, i32, vp, vp]),
            "blake3_tile_count": (u64, [u64, i32]),
            "blake3_keyed_tile_roots": (i32, [vp, u64, u64, vp, i32, i32, vp, vp]),
            "blake3_keyed_tile_roots_ex": (i32, [vp, u64, u64, vp, i32, i32, vp, vp, vp]),
            "blake3_reduce_workspace_size": (sz, [u64, i32]),
            "blake3_keyed_reduce_cvs": (i32, [vp, u64, vp, i32, i32, vp, vp, sz, vp]),
            "blake3_device_status": (i32, [ctypes.POINTER(ctypes.c_uint32)]),
            "blake3_selftest_bounded_wait": (i32, [ctypes.c_uint32, ctypes.POINTER(ctypes.c_int)]),
            "blake3_selftest_compress_rate": (i32, [ctypes.c_uint32, ctypes.c_uint32, vp, vp]),
            "blake3_keyed_hash_xof": (i32, [vp, u64, vp, vp, u64, vp]),
            "blake3_hasher_new": (i32, [vp, ctypes.POINTER(vp)]),
            "blake3_hasher_free": (None, [vp]),
            "blake3_hasher_reset": (i32, [vp]),
            "blake3_hasher_count": (u64, [vp]),
            "blake3_hasher_update": (i32, [vp, vp, u64, vp]),
            "blake3_hasher_update_many": (i32, [vp, vp, vp, u64, vp]),
            "blake3_hasher_export_size": (sz, [vp]),
            "blake3_hasher_export": (i32, [vp, vp, sz, vp]),
            "blake3_hasher_import": (i32, [vp, sz, ctypes.POINTER(vp), vp]),
            "blake3_hasher_finalize": (i32, [vp, vp, u64, vp]),
            "blake3_keyed_hash_host": (i32, [vp, u64, vp, vp, vp, sz, vp]),
            "blake3_hash": (i32, [vp, u64, vp, vp]),
            "blake3_hash_ws": (i32, [vp, u64, vp, vp, sz, vp]),
            "blake3_hash_xof": (i32, [vp, u64, vp, u64, vp]),
            "blake3_hasher_new_default": (i32, [ctypes.POINTER(vp)]),
            "blake3_hash_host": (i32, [vp, u64, vp, vp, sz, vp]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int, where: str) -> None:
    if status != B3G_OK:
        detail = library().blake3_last_cuda_error().decode() if status == 4 else ""
        raise B3GError(status, where, detail)


def _dev_ptr(t: torch.Tensor | None, what: str):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr() if t.numel() else None


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _key(key) -> bytes:
    key = bytes(key)
    if len(key) != 32:
        raise ValueError("key must be 32 bytes")
    return key


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _out32(out: torch.Tensor | None, like: torch.Tensor | None) -> torch.Tensor:
    if out is None:
        dev = like.device if like is not None and like.is_cuda else torch.device("cuda")
        out = torch.empty(32, dtype=torch.uint8, device=dev)
    if _nbytes(out) < 32:
        raise ValueError("output needs 32 bytes")
    return out


def blake3_strerror(status: int) -> str:
    return library().blake3_strerror(status).decode()


def blake3_workspace_size(nbytes: int) -> int:
    return int(library().blake3_workspace_size(nbytes))


def blake3_reduce_workspace_size(count: int, group_log2: int = -1) -> int:
    return int(library().blake3_reduce_workspace_size(count, group_log2))


def blake3_keyed_hash(data: torch.Tensor, key, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Digest of the bytes of the contiguous CUDA tensor `data` (32-byte uint8 tensor)."""
    out = _out32(out, data)
    st = library().blake3_keyed_hash(_dev_ptr(data, "data"), _nbytes(data), _key(key), _dev_ptr(out, "out"),
                                     _stream(stream))
    _check(st, "blake3_keyed_hash")
    return out


def blake3_keyed_hash_ws(data: torch.Tensor, key, workspace: torch.Tensor | None,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out = _out32(out, data)
    ws_ptr = _dev_ptr(workspace, "workspace") if workspace is not None else None
    ws_bytes = _nbytes(workspace) if workspace is not None else 0
    st = library().blake3_keyed_hash_ws(_dev_ptr(data, "data"), _nbytes(data), _key(key), _dev_ptr(out, "out"),
                                        ws_ptr, ws_bytes, _stream(stream))
    _check(st, "blake3_keyed_hash_ws")
    return out


def blake3_keyed_hash_ex(data: torch.Tensor, key, status: torch.Tensor, workspace: torch.Tensor | None = None,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Keyed digest whose kernels report a given-up wait in `status` (a CUDA int32/uint32
    word the caller owns and zeroes), in stream order."""
    out = _out32(out, data)
    ws_ptr = _dev_ptr(workspace, "workspace") if workspace is not None else None
    ws_bytes = _nbytes(workspace) if workspace is not None else 0
    st = library().blake3_keyed_hash_ex(_dev_ptr(data, "data"), _nbytes(data), _key(key), _dev_ptr(out, "out"),
                                        ws_ptr, ws_bytes, _dev_ptr(status, "status"), _stream(stream))
    _check(st, "blake3_keyed_hash_ex")
    return out


def blake3_hash(data: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Default-mode (unkeyed) digest of the contiguous CUDA tensor `data`."""
    out = _out32(out, data)
    st = library().blake3_hash(_dev_ptr(data, "data"), _nbytes(data), _dev_ptr(out, "out"), _stream(stream))
    _check(st, "blake3_hash")
    return out


def blake3_hash_ws(data: torch.Tensor, workspace: torch.Tensor | None, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    out = _out32(out, data)
    ws_ptr = _dev_ptr(workspace, "workspace") if workspace is not None else None
    ws_bytes = _nbytes(workspace) if workspace is not None else 0
    st = library().blake3_hash_ws(_dev_ptr(data, "data"), _nbytes(data), _dev_ptr(out, "out"), ws_ptr, ws_bytes,
                                  _stream(stream))
    _check(st, "blake3_hash_ws")
    return out


def blake3_keyed_hash_noalloc(data: torch.Tensor, key, out: torch.Tensor, stream=None) -> torch.Tensor:
    """The digest without any device allocation: for callers that cannot allocate at
    hashing time.  Uses the library's fixed scratch array (inputs up to 16 GiB); calls
    that overlap on the GPU race on that array, so serialise them."""
    st = library().blake3_keyed_hash_noalloc(_dev_ptr(data, "data"), _nbytes(data), _key(key),
                                             _dev_ptr(out, "out"), _stream(stream))
    _check(st, "blake3_keyed_hash_noalloc")
    return out


def blake3_keyed_chunk_cvs(data: torch.Tensor, key, chunk_offset: int = 0, out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """All chunk CVs as a (n_chunks, 32) uint8 CUDA tensor."""
    n = max(1, -(-_nbytes(data) // 1024))
    if out is None:
        out = torch.empty((n, 32), dtype=torch.uint8, device=data.device)
    if _nbytes(out) < 32 * n:
        raise ValueError("chunk CV output too small")
    st = library().blake3_keyed_chunk_cvs(_dev_ptr(data, "data"), _nbytes(data), chunk_offset, _key(key),
                                          _dev_ptr(out, "out"), _stream(stream))
    _check(st, "blake3_keyed_chunk_cvs")
    return out


def blake3_keyed_subtree_root(data: torch.Tensor, key, chunk_offset: int = 0, is_root: bool = False,
                              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out = _out32(out, data)
    st = library().blake3_keyed_subtree_root(_dev_ptr(data, "data"), _nbytes(data), chunk_offset, _key(key),
                                             int(is_root), _dev_ptr(out, "out"), _stream(stream))
    _check(st, "blake3_keyed_subtree_root")
    return out


def blake3_tile_count(nbytes: int, leaves_log2: int = -1) -> int:
    return int(library().blake3_tile_count(nbytes, leaves_log2))


def blake3_keyed_tile_roots(data: torch.Tensor, key, chunk_offset: int = 0, leaves_log2: int = -1,
                            is_root: bool = False, out: torch.Tensor | None = None, stream=None,
                            tile_counter: torch.Tensor | None = None) -> torch.Tensor:
    """CTA subtree roots as a (tiles, 32) uint8 CUDA tensor.  With `tile_counter` (a CUDA
    word the caller has zeroed on the stream) the tiles are scheduled dynamically
    (blake3_keyed_tile_roots_ex)."""
    tiles = blake3_tile_count(_nbytes(data), leaves_log2)
    if tiles == 0:
        raise B3GError(6, "blake3_keyed_tile_roots", "leaves_log2 out of range")
    if out is None:
        out = torch.empty((tiles, 32), dtype=torch.uint8, device=data.device)
    if _nbytes(out) < 32 * tiles:
        raise ValueError("tile root output too small")
    st = library().blake3_keyed_tile_roots_ex(_dev_ptr(data, "data"), _nbytes(data), chunk_offset, _key(key),
                                              leaves_log2, int(is_root), _dev_ptr(out, "out"),
                                              _dev_ptr(tile_counter, "tile_counter"), _stream(stream))
    _check(st, "blake3_keyed_tile_roots_ex")
    return out


def blake3_keyed_reduce_cvs(cvs: torch.Tensor, key, is_root: bool = False, group_log2: int = -1,
                            out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """Reduce a (count, 32) uint8 CUDA tensor of subtree CVs to one CV."""
    count = _nbytes(cvs) // 32
    out = _out32(out, cvs)
    if workspace is None:
        need = blake3_reduce_workspace_size(count, group_log2) if count else 0
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=cvs.device)
    st = library().blake3_keyed_reduce_cvs(_dev_ptr(cvs, "cvs"), count, _key(key), int(is_root), group_log2,
                                           _dev_ptr(out, "out"), _dev_ptr(workspace, "workspace"),
                                           _nbytes(workspace), _stream(stream))
    _check(st, "blake3_keyed_reduce_cvs")
    return out


def blake3_device_status() -> int:
    v = ctypes.c_uint32(0)
    _check(library().blake3_device_status(ctypes.byref(v)), "blake3_device_status")
    return int(v.value)


def blake3_selftest_bounded_wait(limit_us: int) -> bool:
    flag = ctypes.c_int(-1)
    _check(library().blake3_selftest_bounded_wait(limit_us, ctypes.byref(flag)), "blake3_selftest_bounded_wait")
    return flag.value == 1


def blake3_selftest_bounded_wait_ex(limit_us: int, status: torch.Tensor, stream=None) -> None:
    """The bounded-wait probe on `stream`, ORing the timeout bit into the device word `status`."""
    _check(library().blake3_selftest_bounded_wait_ex(limit_us, _dev_ptr(status, "status"), _stream(stream)),
           "blake3_selftest_bounded_wait_ex")


def blake3_selftest_compress_latency(lanes_per_chunk: int, chain: int, key, cvs: torch.Tensor,
                                     cycles: torch.Tensor, stream=None) -> None:
    """One warp of compression chains with 1 or 4 lanes per chain (asynchronous): the chains'
    final CVs into `cvs` (32 / lanes_per_chunk x 32 bytes) and lane 0's cycles into `cycles`
    (an int64 CUDA tensor)."""
    _check(library().blake3_selftest_compress_latency(lanes_per_chunk, chain, _key(key), _dev_ptr(cvs, "cvs"),
                                                      _dev_ptr(cycles, "cycles"), _stream(stream)),
           "blake3_selftest_compress_latency")


def blake3_selftest_compress_rate(blocks: int, iters: int, sink: torch.Tensor, stream=None) -> None:
    """Launch blocks x 128 threads of `iters` chained compressions each (no memory traffic
    but the 4-byte `sink`), asynchronously on `stream`: the compression-only ceiling."""
    _check(library().blake3_selftest_compress_rate(blocks, iters, _dev_ptr(sink, "sink"), _stream(stream)),
           "blake3_selftest_compress_rate")


def blake3_keyed_hash_xof(data: torch.Tensor, key, out_len: int, out: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """out_len bytes of extendable output (a uint8 CUDA tensor); the first 32 are the digest."""
    if out is None:
        dev = data.device if data.is_cuda else torch.device("cuda")
        out = torch.empty(out_len, dtype=torch.uint8, device=dev)
    if _nbytes(out) < out_len:
        raise ValueError("output too small")
    st = library().blake3_keyed_hash_xof(_dev_ptr(data, "data"), _nbytes(data), _key(key),
                                         _dev_ptr(out, "out") if out_len else None, out_len, _stream(stream))
    _check(st, "blake3_keyed_hash_xof")
    return out


def blake3_hash_xof(data: torch.Tensor, out_len: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out_len bytes of default-mode (unkeyed) extendable output."""
    if out is None:
        dev = data.device if data.is_cuda else torch.device("cuda")
        out = torch.empty(out_len, dtype=torch.uint8, device=dev)
    if _nbytes(out) < out_len:
        raise ValueError("output too small")
    st = library().blake3_hash_xof(_dev_ptr(data, "data"), _nbytes(data), _dev_ptr(out, "out") if out_len else None,
                                   out_len, _stream(stream))
    _check(st, "blake3_hash_xof")
    return out


class Hasher:
    """Streaming hasher over device segments (blake3_hasher_* of the C ABI): keyed with
    `key`, or in the default (unkeyed) mode when `key` is None."""

    def __init__(self, key=None):
        self._h = ctypes.c_void_p()
        if key is None:
            _check(library().blake3_hasher_new_default(ctypes.byref(self._h)), "blake3_hasher_new_default")
        else:
            _check(library().blake3_hasher_new(_key(key), ctypes.byref(self._h)), "blake3_hasher_new")

    def update(self, data: torch.Tensor, stream=None) -> "Hasher":
        _check(library().blake3_hasher_update(self._h, _dev_ptr(data, "data"), _nbytes(data), _stream(stream)),
               "blake3_hasher_update")
        return self

    def update_many(self, segments, stream=None) -> "Hasher":
        """Absorb a sequence of contiguous CUDA tensors in order, as one call (runs of small
        segments are copied by one gather launch)."""
        segs = list(segments)
        n = len(segs)
        ptrs = (ctypes.c_void_p * max(1, n))(*[_dev_ptr(t, "segment") for t in segs])
        lens = (ctypes.c_uint64 * max(1, n))(*[_nbytes(t) for t in segs])
        _check(library().blake3_hasher_update_many(self._h, ptrs, lens, n, _stream(stream)),
               "blake3_hasher_update_many")
        return self

    def finalize(self, out_len: int = 32, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty(max(out_len, 1), dtype=torch.uint8, device="cuda")[:out_len]
        _check(library().blake3_hasher_finalize(self._h, _dev_ptr(out, "out") if out_len else None, out_len,
                                                _stream(stream)), "blake3_hasher_finalize")
        return out

    def reset(self) -> "Hasher":
        _check(library().blake3_hasher_reset(self._h), "blake3_hasher_reset")
        return self

    @property
    def count(self) -> int:
        return int(library().blake3_hasher_count(self._h))

    def export(self, stream=None) -> bytes:
        """The hasher's whole state as bytes (checkpoint); the hasher is not changed."""
        n = library().blake3_hasher_export_size(self._h)
        buf = ctypes.create_string_buffer(max(1, n))
        _check(library().blake3_hasher_export(self._h, buf, n, _stream(stream)), "blake3_hasher_export")
        return buf.raw[:n]

    @classmethod
    def from_state(cls, state: bytes, stream=None) -> "Hasher":
        """A hasher on the current device resumed from Hasher.export() bytes."""
        self = cls.__new__(cls)
        self._h = ctypes.c_void_p()
        buf = ctypes.create_string_buffer(bytes(state), len(state))
        _check(library().blake3_hasher_import(buf, len(state), ctypes.byref(self._h), _stream(stream)),
               "blake3_hasher_import")
        return self

    def close(self) -> None:
        if self._h:
            library().blake3_hasher_free(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def blake3_keyed_hash_host(data: torch.Tensor, key, staging: torch.Tensor | None = None, stream=None) -> bytes:
    """Digest of a contiguous HOST tensor (pinned for full speed), copied and hashed in
    overlapping segments; returns the 32 digest bytes."""
    if data.is_cuda:
        raise ValueError("data must be a host tensor")
    t = data.contiguous()
    out = ctypes.create_string_buffer(32)
    st_ptr = _dev_ptr(staging, "staging") if staging is not None else None
    st_bytes = _nbytes(staging) if staging is not None else 0
    st = library().blake3_keyed_hash_host(t.data_ptr() if t.numel() else None, _nbytes(t), _key(key), out,
                                          st_ptr, st_bytes, _stream(stream))
    _check(st, "blake3_keyed_hash_host")
    return out.raw


def blake3_hash_host(data: torch.Tensor, staging: torch.Tensor | None = None, stream=None) -> bytes:
    """Default-mode (unkeyed) digest of a contiguous HOST tensor; see blake3_keyed_hash_host."""
    if data.is_cuda:
        raise ValueError("data must be a host tensor")
    t = data.contiguous()
    out = ctypes.create_string_buffer(32)
    st_ptr = _dev_ptr(staging, "staging") if staging is not None else None
    st_bytes = _nbytes(staging) if staging is not None else 0
    st = library().blake3_hash_host(t.data_ptr() if t.numel() else None, _nbytes(t), out, st_ptr, st_bytes,
                                    _stream(stream))
    _check(st, "blake3_hash_host")
    return out.raw


B3G_OPT_FUSED_FINAL = 1
B3G_OPT_FAIL_ALLOC = 2
B3G_OPT_STREAM_UNBATCHED = 3


def blake3_set_option(option: int, value: int) -> None:
    _check(library().blake3_set_option(option, value), "blake3_set_option")

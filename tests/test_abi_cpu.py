"""The C-ABI library without a GPU: it loads, exports every declared symbol, and its
host-side logic (sizes, argument checks that return before any CUDA call) works."""

import ctypes
import glob
import os
import re

import pytest

from blake3_merkle_tree_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails its checks first
KEY = bytes(range(32))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if m.group(1) not in ("defined",):
                names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from blake3_merkle_tree_gb300 import build

    build.build()
    return binding.library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "blake3_keyed_hash" in names and len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_strerror(lib):
    for code in range(7):
        assert lib.blake3_strerror(code)
    assert lib.blake3_strerror(99) == b"unknown status"


def test_sizes(lib):
    assert lib.blake3_default_leaves_log2() == 7
    assert lib.blake3_tile_count(0, -1) == 1
    assert lib.blake3_tile_count(128 * 1024, -1) == 1
    assert lib.blake3_tile_count(128 * 1024 + 1, -1) == 2
    assert lib.blake3_tile_count(12 * (1 << 30) + 777, 8) == 49153
    assert lib.blake3_tile_count(12 * (1 << 30) + 777, -1) == 98305
    assert lib.blake3_tile_count(1 << 20, 5) == 32
    assert lib.blake3_tile_count(1 << 20, 4) == 0
    assert lib.blake3_workspace_size(0) == 0  # one chunk, one tile: no workspace
    assert lib.blake3_workspace_size(32 * 1024) == 0  # 32 chunks fit one 32-chunk tile
    # small inputs spread over 32-chunk tiles: 1 MiB = 1024 chunks = 32 tiles, reduced by
    # the last CTA (16 bytes for its ticket counter)
    assert lib.blake3_workspace_size(1 << 20) == 32 * 32 + 16
    assert lib.blake3_workspace_size(256 * 1024) == 8 * 32 + 16
    # up to 32,768 tile CVs the reduction takes groups of 64: 64 MiB = 65536 chunks,
    # 128-chunk tiles already give 512 CTAs, reduced 512 -> 8 -> 1
    assert lib.blake3_workspace_size(64 << 20) == 512 * 32 + 8 * 32
    assert lib.blake3_workspace_size(19 << 20) == 152 * 32 + 3 * 32  # 19456 chunks / 128
    # 144 tiles of 128: fewer than one per SM, but at least 80 keep 128-chunk tiles,
    # 144 -> 3 -> 1 (10 MiB: 80 -> 2 -> 1); below 80 (9 MiB: 72) the tiles shrink until
    # there are 152: 32 chunks, 288 -> 5 -> 1
    assert lib.blake3_workspace_size(18 << 20) == 144 * 32 + 3 * 32
    assert lib.blake3_workspace_size(10 << 20) == 80 * 32 + 2 * 32
    assert lib.blake3_workspace_size(9 << 20) == 288 * 32 + 5 * 32
    # 4 GiB: 32768 tile CVs, then 512 and 8 group CVs, then 16 bytes for the tile counter
    # (more tiles than one per resident CTA)
    assert lib.blake3_workspace_size(1 << 32) == 32768 * 32 + 512 * 32 + 8 * 32 + 16
    # 12 GiB + 777: 98305 tile CVs, groups of 1024 above 32,768 CVs: 97 group CVs
    assert lib.blake3_workspace_size(12 * (1 << 30) + 777) == 98305 * 32 + 97 * 32 + 16
    # 760 tiles of 128 chunks: no counter; 761: a counter
    assert lib.blake3_workspace_size(760 * 128 * 1024) == 760 * 32 + 12 * 32
    assert lib.blake3_workspace_size(760 * 128 * 1024 + 1) == 761 * 32 + 12 * 32 + 16
    assert lib.blake3_reduce_workspace_size(1024, 10) == 0
    assert lib.blake3_reduce_workspace_size(1025, 10) == 64
    assert lib.blake3_reduce_workspace_size(5, 1) == 3 * 32 + 32 + 32
    assert lib.blake3_reduce_workspace_size(64, -1) == 0
    assert lib.blake3_reduce_workspace_size(2048, -1) == 32 * 32
    assert lib.blake3_reduce_workspace_size(32768, -1) == 512 * 32 + 8 * 32
    assert lib.blake3_reduce_workspace_size(32769, -1) == 33 * 32


def test_compress_rate_selftest_checks_arguments_first(lib):
    f = lib.blake3_selftest_compress_rate
    f.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(1, 1, None, None) == 1  # no sink
    assert f(0, 1, FAKE, None) == 6 and f(1, 0, FAKE, None) == 6  # empty launch
    assert f((1 << 20) + 1, 1, FAKE, None) == 6 and f(1, (1 << 20) + 1, FAKE, None) == 6
    assert f(1, 1, ctypes.c_void_p(0x10002), None) == 2  # sink not 4-byte aligned


def test_argument_errors_before_any_cuda_call(lib):
    out = FAKE
    assert lib.blake3_keyed_hash(FAKE, 10, None, out, None) == 1
    assert lib.blake3_keyed_hash(None, 10, KEY, out, None) == 1
    assert lib.blake3_keyed_hash(FAKE, 10, KEY, None, None) == 1
    assert lib.blake3_keyed_hash_ws(FAKE, 1 << 30, KEY, out, None, 0, None) == 3
    assert lib.blake3_keyed_hash_ws(FAKE, 1 << 30, KEY, out, FAKE, 16, None) == 3
    assert lib.blake3_keyed_hash_ws(FAKE, 1 << 30, KEY, out, ctypes.c_void_p(0x10001), 1 << 20, None) == 2
    assert lib.blake3_keyed_subtree_root(FAKE, 4 * 1024, 2, KEY, 0, out, None) == 2
    assert lib.blake3_keyed_subtree_root(FAKE, 3 * 1024, 6, KEY, 0, out, None) == 2
    assert lib.blake3_keyed_tile_roots(FAKE, 4096, 0, KEY, 9, 0, out, None) == 6
    assert lib.blake3_keyed_tile_roots(FAKE, 4096, 0, KEY, 4, 0, out, None) == 6
    assert lib.blake3_keyed_reduce_cvs(FAKE, 0, KEY, 0, -1, out, FAKE, 0, None) == 6
    assert lib.blake3_keyed_reduce_cvs(FAKE, 1, KEY, 1, -1, out, FAKE, 0, None) == 6
    assert lib.blake3_keyed_reduce_cvs(FAKE, 8, KEY, 1, 11, out, FAKE, 0, None) == 6
    assert lib.blake3_keyed_reduce_cvs(FAKE, 5000, KEY, 1, 10, out, None, 0, None) == 3
    assert lib.blake3_keyed_chunk_cvs(FAKE, 10, 0, KEY, None, None) == 1
    assert lib.blake3_device_status(None) == 1
    assert lib.blake3_selftest_bounded_wait(0, ctypes.byref(ctypes.c_int())) == 6
    assert lib.blake3_selftest_bounded_wait(10, None) == 1
    ex = lib.blake3_keyed_hash_ex
    assert ex(FAKE, 10, KEY, FAKE, None, 0, None, None) == 1  # no status word
    assert ex(FAKE, 10, KEY, FAKE, None, 0, ctypes.c_void_p(0x10002), None) == 2  # status not 4-byte aligned
    assert ex(FAKE, 1 << 30, KEY, FAKE, FAKE, 16, FAKE, None) == 3  # workspace too small
    assert lib.blake3_selftest_bounded_wait_ex(10, None, None) == 1
    assert lib.blake3_selftest_bounded_wait_ex(0, FAKE, None) == 6
    assert lib.blake3_selftest_bounded_wait_ex(10, ctypes.c_void_p(0x10001), None) == 2


def test_binding_refuses_host_tensors(lib):
    import torch

    with pytest.raises(ValueError):
        binding.blake3_keyed_hash(torch.zeros(10, dtype=torch.uint8), KEY, out=torch.zeros(32, dtype=torch.uint8))


def test_output_alignment_is_checked(lib):
    odd = ctypes.c_void_p(0x10008)
    assert lib.blake3_keyed_hash(FAKE, 10, KEY, odd, None) == 2
    assert lib.blake3_keyed_hash_ws(FAKE, 10, KEY, odd, None, 0, None) == 2
    assert lib.blake3_keyed_chunk_cvs(FAKE, 10, 0, KEY, odd, None) == 2
    assert lib.blake3_keyed_subtree_root(FAKE, 10, 0, KEY, 1, odd, None) == 2
    assert lib.blake3_keyed_tile_roots(FAKE, 10, 0, KEY, -1, 1, odd, None) == 2
    assert lib.blake3_keyed_reduce_cvs(odd, 4, KEY, 1, -1, FAKE, FAKE, 0, None) == 2


def test_stream_and_xof_argument_errors(lib):
    h = ctypes.c_void_p()
    assert lib.blake3_hasher_new(None, ctypes.byref(h)) == 1
    assert lib.blake3_hasher_new(KEY, None) == 1
    assert lib.blake3_hasher_update(None, FAKE, 10, None) == 1
    assert lib.blake3_hasher_finalize(None, FAKE, 32, None) == 1
    assert lib.blake3_hasher_reset(None) == 1
    assert lib.blake3_hasher_count(None) == 0
    lib.blake3_hasher_free(None)
    assert lib.blake3_keyed_hash_xof(FAKE, 10, None, FAKE, 32, None) == 1
    assert lib.blake3_hasher_update_many(None, FAKE, FAKE, 1, None) == 1
    assert lib.blake3_hasher_update_many(FAKE, None, FAKE, 1, None) == 1
    assert lib.blake3_hasher_update_many(FAKE, FAKE, None, 1, None) == 1
    assert lib.blake3_keyed_hash_xof(FAKE, 10, KEY, None, 32, None) == 1


def test_host_entry_argument_errors(lib):
    out = ctypes.create_string_buffer(32)
    assert lib.blake3_keyed_hash_host(FAKE, 10, None, out, None, 0, None) == 1
    assert lib.blake3_keyed_hash_host(FAKE, 10, KEY, None, None, 0, None) == 1
    assert lib.blake3_keyed_hash_host(None, 10, KEY, out, None, 0, None) == 1


def test_default_mode_argument_errors(lib):
    out = ctypes.create_string_buffer(32)
    odd = ctypes.c_void_p(0x10008)
    assert lib.blake3_hash(None, 10, FAKE, None) == 1
    assert lib.blake3_hash(FAKE, 10, None, None) == 1
    assert lib.blake3_hash(FAKE, 10, odd, None) == 2
    assert lib.blake3_hash_ws(FAKE, 1 << 30, FAKE, None, 0, None) == 3
    assert lib.blake3_hash_ws(FAKE, 1 << 30, FAKE, ctypes.c_void_p(0x10001), 1 << 20, None) == 2
    assert lib.blake3_hash_ws(FAKE, 10, odd, None, 0, None) == 2
    assert lib.blake3_hash_xof(None, 10, FAKE, 32, None) == 1
    assert lib.blake3_hash_xof(FAKE, 10, None, 32, None) == 1
    assert lib.blake3_hasher_new_default(None) == 1
    assert lib.blake3_hash_host(None, 10, out, None, 0, None) == 1
    assert lib.blake3_hash_host(FAKE, 10, None, None, 0, None) == 1
    # the workspace of the default mode is the keyed mode's
    assert lib.blake3_workspace_size(1 << 30) > 0


def test_options_and_config(lib):
    assert lib.blake3_set_option(99, 1) == 6
    assert lib.blake3_set_option(2, -1) == 6  # the allocation-failure hook takes n >= 0
    assert lib.blake3_set_option(2, 0) == 0
    assert lib.blake3_set_option(3, 1) == 0 and lib.blake3_set_option(3, 0) == 0
    assert lib.blake3_set_option(1, 0) == 0
    assert lib.blake3_kernel_config().startswith((b"leaf_async_kernel<", b"leaf_tma_kernel<"))


def _state_record(magic=0x48473342, version=1, mode=16, depth=1, count=3000, pushed=2, acc_len=952,
                  extra=0):
    import struct

    head = struct.pack("<4I", magic, version, mode, depth) + bytes(32) + struct.pack("<3Q", count, pushed, acc_len)
    return head + bytes(32 * depth + acc_len + extra)


def test_hasher_import_rejects_bad_records_before_any_cuda_call(lib):
    h = ctypes.c_void_p()

    def imp(rec, size=None):
        buf = ctypes.create_string_buffer(rec, len(rec))
        return lib.blake3_hasher_import(buf, len(rec) if size is None else size, ctypes.byref(h), None)

    assert lib.blake3_hasher_import(None, 100, ctypes.byref(h), None) == 1
    assert lib.blake3_hasher_import(FAKE, 100, None, None) == 1
    assert imp(_state_record(), size=20) == 6                     # shorter than the header
    assert imp(_state_record(magic=0x12345678)) == 6              # not a hasher record
    assert imp(_state_record(version=2)) == 6                     # unknown version
    assert imp(_state_record(mode=32)) == 6                       # unknown hash mode
    assert imp(_state_record(count=3001)) == 6                    # count != pushed * 1024 + buffered
    assert imp(_state_record(depth=0)) == 6                       # pushed chunks but an empty stack
    assert imp(_state_record(depth=70)) == 6                      # deeper than the stack
    assert imp(_state_record(count=1024, pushed=1, acc_len=0)) == 6  # one chunk is never pushed
    assert imp(_state_record(acc_len=(64 << 20) + 1, count=2048 + (64 << 20) + 1)) == 6  # buffer too large
    rec = _state_record()
    assert imp(rec, size=len(rec) - 1) == 6                       # truncated stack or bytes
    assert lib.blake3_hasher_export_size(None) == 0
    assert lib.blake3_hasher_export(None, FAKE, 100, None) == 1

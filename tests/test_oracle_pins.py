"""Pins of the CPU oracle against things other than itself (CPU only).

What each test pins:
  * IV                    - closed form: first 32 bits of the fractional parts of
                            the square roots of the first eight primes.
  * G, rotations, column/diagonal word assignment, IV
                          - the oracle's round function, driven with the BLAKE2s
                            schedule of RFC 7693, must reproduce hashlib.blake2s.
  * tree shape            - recursive largest-power-of-two split == stack merge on
                            every length 0..65536 ("BLAKE3 GPU 400x faster hashing",
                            section "BLAKE3": left subtree full and left-large);
                            the page's worked example 13 = 8 + 4 + 1 (section
                            "Merkle Tree 归约"), read from tests/golden.
  * ROOT placement        - a one-chunk input equals its block chain with ROOT on
                            the last block only (section "Kernel 2 和 3": ROOT on
                            the final compression).
  * tile decomposition    - the digest does not depend on the tile size 2^t
                            (section "Kernel 1": t is a free parameter).
The BLAKE3 message permutation, flag values, state layout and round count have
no known-answer source here; they are checked for consistency only
(parity unpinned).
"""

import hashlib
import math
import os
import re

import numpy as np
import pytest

import oracle
from blake3_merkle_tree_gb300 import workloads

HERE = os.path.dirname(os.path.abspath(__file__))
KEY = workloads.key_bytes(1)


def _data(n, seed=12345):
    return workloads.numpy_uniform_bytes(seed, n)


def test_iv_closed_form():
    primes = [2, 3, 5, 7, 11, 13, 17, 19]
    # floor(frac(sqrt(p)) * 2^32) == isqrt(p * 2^64) mod 2^32
    expected = [math.isqrt(p << 64) & 0xFFFFFFFF for p in primes]
    assert oracle.iv() == expected


@pytest.mark.parametrize("n", [0, 1, 3, 55, 63, 64, 65, 127, 128, 129, 191, 1000, 1024, 4099])
def test_round_function_reproduces_blake2s(n):
    msg = _data(n, seed=77 + n).tobytes()
    assert oracle.blake2s_256(msg) == hashlib.blake2s(msg).digest()


def test_blake2s_pin_detects_a_planted_mistake(tmp_path):
    """A wrong rotation or word index in the round function must break the pin."""
    import ctypes
    import subprocess

    src = open(os.path.join(os.path.dirname(oracle.__file__), "blake3_oracle.c")).read()
    mutants = {
        "rot12": src.replace("rotr32(v[b] ^ v[c], 12)", "rotr32(v[b] ^ v[c], 11)"),
        "diag": src.replace("g(v, 1, 6, 11, 12, s[10], s[11]);", "g(v, 1, 6, 11, 13, s[10], s[11]);"),
        "iv": src.replace("0x9B05688Cu", "0x9B05688Du"),
        "drop_y": src.replace("v[a] = v[a] + v[b] + y;", "v[a] = v[a] + v[b];"),
    }
    msg = _data(200, seed=5).tobytes()
    good = hashlib.blake2s(msg).digest()
    for name, text in mutants.items():
        assert text != src, name
        c = tmp_path / f"{name}.c"
        so = tmp_path / f"{name}.so"
        c.write_text(text)
        subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(c)], check=True)
        lib = ctypes.CDLL(str(so))
        out = ctypes.create_string_buffer(32)
        lib.oracle_blake2s_256(msg, ctypes.c_size_t(len(msg)), out)
        assert out.raw != good, f"mutant {name} was not caught"


def test_permutation_and_flags_are_consistent():
    perm = oracle.msg_permutation()
    assert sorted(perm) == list(range(16))
    f = oracle.flags()
    bits = list(f.values())
    assert all(b and (b & (b - 1)) == 0 for b in bits)
    assert len(set(bits)) == 5


@pytest.mark.slow
def test_recursive_equals_stack_every_length_to_64KiB():
    buf = _data(65536, seed=2024)
    for n in range(0, 65537):
        a = oracle.keyed_hash(buf[:n], KEY)
        b = oracle.keyed_hash_recursive(buf[:n], KEY)
        assert a == b, n


def _eval_shape(expr, chunks_cv, key, root=True):
    tokens = re.findall(r"P\(|C\d+|\)|,", expr)
    pos = 0

    def node(is_root):
        nonlocal pos
        tok = tokens[pos]
        pos += 1
        if tok.startswith("C"):
            return chunks_cv[int(tok[1:])]
        assert tok == "P("
        left = node(False)
        assert tokens[pos] == ","
        pos += 1
        right = node(False)
        assert tokens[pos] == ")"
        pos += 1
        return oracle.parent_cv(key, left, right, is_root)

    out = node(root)
    assert pos == len(tokens)
    return out


def test_thirteen_leaf_example_from_the_page():
    text = open(os.path.join(HERE, "golden", "tree_13_leaves.txt")).read()
    expr = [ln for ln in text.splitlines() if ln and not ln.startswith("#")][0].strip()
    data = _data(13 * 1024, seed=13)
    cvs = [oracle.chunk_cv(KEY, data[i * 1024:(i + 1) * 1024], i) for i in range(13)]
    assert _eval_shape(expr, cvs, KEY) == oracle.keyed_hash(data, KEY)
    assert _eval_shape(expr, cvs, KEY) == oracle.keyed_hash_recursive(data, KEY)
    # and the chunk CVs agree with the bulk entry point
    bulk = oracle.chunk_cvs(data, KEY)
    assert [bytes(r) for r in bulk] == cvs


@pytest.mark.parametrize("n", [0, 1, 2, 63, 64, 65, 127, 128, 500, 960, 1023, 1024])
def test_one_chunk_identity(n):
    """len <= 1024: the digest is the block chain of the single chunk, ROOT on its last block."""
    f = oracle.flags()
    data = _data(n, seed=300 + n).tobytes()
    nblocks = max(1, -(-n // 64))
    cv = KEY
    for b in range(nblocks):
        part = data[64 * b:64 * (b + 1)]
        flags = f["KEYED_HASH"]
        if b == 0:
            flags |= f["CHUNK_START"]
        if b == nblocks - 1:
            flags |= f["CHUNK_END"] | f["ROOT"]
        cv = oracle.compress(cv, part.ljust(64, b"\0"), 0, len(part), flags)[:32]
    assert cv == oracle.keyed_hash(data, KEY)
    assert cv == oracle.chunk_cv(KEY, data, 0, is_root=True)
    # the same chunk without ROOT is a different value
    assert oracle.chunk_cv(KEY, data, 0, is_root=False) != cv


def _fold_tiles(tile_cvs, key, is_root):
    n = len(tile_cvs)
    if n == 1:
        return tile_cvs[0]
    p = 1
    while p * 2 < n:
        p *= 2
    left = _fold_tiles(tile_cvs[:p], key, False)
    right = _fold_tiles(tile_cvs[p:], key, False)
    return oracle.parent_cv(key, left, right, is_root)


@pytest.mark.parametrize("length", [1024, 2049, 13 * 1024, 13 * 1024 + 7, 33 * 1024, 100 * 1024 + 5,
                                    257 * 1024, 300 * 1024 - 1])
def test_digest_independent_of_tile_size(length):
    data = _data(length, seed=length)
    ref = oracle.keyed_hash(data, KEY)
    nchunks = max(1, -(-length // 1024))
    for t in range(0, 10):
        tile = 1 << t
        ntiles = -(-nchunks // tile)
        if ntiles == 1:
            got = oracle.subtree_cv(data, KEY, 0, is_root=True)
        else:
            tiles = [oracle.subtree_cv(data[i * tile * 1024:(i + 1) * tile * 1024], KEY, i * tile)
                     for i in range(ntiles)]
            got = _fold_tiles(tiles, KEY, True)
        assert got == ref, (length, t)


def test_root_flag_only_on_final_compression():
    data = _data(5 * 1024, seed=9)
    with_root = oracle.keyed_hash(data, KEY)
    no_root = oracle.subtree_cv(data, KEY, 0, is_root=False)
    assert with_root != no_root
    assert oracle.subtree_cv(data, KEY, 0, is_root=True) == with_root


def test_counter_is_per_chunk():
    """Identical chunk contents at different positions give different CVs."""
    block = _data(1024, seed=4).tobytes()
    a = oracle.chunk_cv(KEY, block, 0)
    b = oracle.chunk_cv(KEY, block, 1)
    c = oracle.chunk_cv(KEY, block, 1 << 32)
    assert len({a, b, c}) == 3
    cvs = oracle.chunk_cvs(np.frombuffer(block * 3, dtype=np.uint8), KEY)
    assert bytes(cvs[0]) == a and bytes(cvs[1]) == b


@pytest.mark.parametrize("length", [0, 1, 64, 1024, 1025, 13 * 1024 + 7, 100 * 1024])
def test_xof_prefix_is_the_digest(length):
    """Extendable output: its first 32 bytes are the digest (the digest is output block 0
    truncated), and a shorter output is a prefix of a longer one."""
    data = _data(length, seed=500 + length)
    digest = oracle.keyed_hash(data, KEY)
    long = oracle.keyed_hash_xof(data, KEY, 1000)
    assert long[:32] == digest
    assert oracle.keyed_hash_xof(data, KEY, 32) == digest
    for n in (0, 1, 63, 64, 65, 200):
        assert oracle.keyed_hash_xof(data, KEY, n) == long[:n]
    # output blocks differ from one another (the counter advances)
    blocks = [long[i:i + 64] for i in range(0, 960, 64)]
    assert len(set(blocks)) == len(blocks)


def test_xof_block_is_the_root_compression_with_counter():
    """Two-chunk input: output block i == compress(key, left||right, i, 64, KEYED|PARENT|ROOT)."""
    f = oracle.flags()
    data = _data(2048, seed=8)
    left = oracle.chunk_cv(KEY, data[:1024], 0)
    right = oracle.chunk_cv(KEY, data[1024:], 1)
    out = oracle.keyed_hash_xof(data, KEY, 64 * 5)
    for i in range(5):
        blk = oracle.compress(KEY, left + right, i, 64, f["KEYED_HASH"] | f["PARENT"] | f["ROOT"])
        assert out[64 * i:64 * (i + 1)] == blk


# ---------------------------------------------------------------------------------
# The default (unkeyed) mode (page section "BLAKE3": the initial chaining value is an
# IV by default, the user's key in keyed mode).  Its IV is pinned by the closed form
# above; its flag word (no mode bit) is unpinned like the other flag values.
# ---------------------------------------------------------------------------------

def _iv_bytes():
    return b"".join(w.to_bytes(4, "little") for w in oracle.iv())


@pytest.mark.parametrize("n", [0, 1, 64, 65, 1023, 1024])
def test_default_mode_one_chunk_identity(n):
    """len <= 1024: the IV-started block chain of the single chunk, no mode bit, ROOT last."""
    f = oracle.flags()
    data = _data(n, seed=700 + n).tobytes()
    cv = _iv_bytes()
    nblocks = max(1, -(-n // 64))
    for b in range(nblocks):
        part = data[64 * b:64 * (b + 1)]
        flags = (f["CHUNK_START"] if b == 0 else 0) | (f["CHUNK_END"] | f["ROOT"] if b == nblocks - 1 else 0)
        cv = oracle.compress(cv, part.ljust(64, b"\0"), 0, len(part), flags)[:32]
    assert cv == oracle.hash(data)


def test_default_mode_tree_forms_agree():
    """Recursive split == stack merge in the default mode on every length class."""
    for n in [0, 1, 1024, 1025, 2048, 3 * 1024 + 1, 8 * 1024, 13 * 1024 + 7, 64 * 1024 - 1, 100 * 1024 + 3]:
        data = _data(n, seed=800 + n).tobytes()
        assert oracle.hash(data) == oracle.hash_recursive(data), n


def test_default_mode_parent_uses_iv_and_no_mode_bit():
    """Two chunks: the root is the parent of the two chunk CVs, started from the IV."""
    f = oracle.flags()
    data = _data(2048, seed=901).tobytes()
    iv = _iv_bytes()

    def chunk(c, ctr):
        cv = iv
        for b in range(16):
            flags = (f["CHUNK_START"] if b == 0 else 0) | (f["CHUNK_END"] if b == 15 else 0)
            cv = oracle.compress(cv, c[64 * b:64 * b + 64], ctr, 64, flags)[:32]
        return cv

    left, right = chunk(data[:1024], 0), chunk(data[1024:], 1)
    root = oracle.compress(iv, left + right, 0, 64, f["PARENT"] | f["ROOT"])[:32]
    assert root == oracle.hash(data)


@pytest.mark.parametrize("n", [0, 5, 1024, 4097])
def test_default_mode_differs_from_keyed_with_iv_key_and_has_xof_prefix(n):
    data = _data(n, seed=950 + n).tobytes()
    assert oracle.hash(data) != oracle.keyed_hash(data, _iv_bytes())  # the mode bit is in every compression
    assert oracle.hash_xof(data, 32) == oracle.hash(data)
    assert oracle.hash_xof(data, 200)[:100] == oracle.hash_xof(data, 100)

"""The C ABI used from a plain C program (no Python between the caller and the library):
its digests, streamed digest, extendable output and host-input digest equal the oracle's."""

import os
import subprocess

import numpy as np
import pytest

import oracle
from blake3_merkle_tree_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "b3g_c_client.c")


@pytest.fixture(scope="module")
def client():
    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = os.path.join(libdir, "_build", "b3g_c_client")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", SRC, "-o", exe,
                    f"-I{os.path.join(ROOT, 'include')}", f"-I{cuda}/include",
                    f"-L{libdir}", "-lb3g", f"-Wl,-rpath,{libdir}", f"-L{cuda}/lib64", "-lcudart",
                    f"-Wl,-rpath,{cuda}/lib64"], check=True)
    return exe


def _inputs(n):
    i = np.arange(n, dtype=np.uint64)
    data = ((131 * i + 7 * (i >> 8) + 3) & 0xFF).astype(np.uint8).tobytes()
    key = bytes((7 * j + 1) & 0xFF for j in range(32))
    return data, key


@pytest.mark.parametrize("n", [0, 1, 1024, 1025, 5 * 1024 * 1024 + 123])
def test_c_client_matches_oracle(client, n):
    p = subprocess.run([client, str(n)], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    one_shot, streamed, xof, from_host, default_mode, status = p.stdout.split()
    data, key = _inputs(n)
    ref = oracle.keyed_hash(data, key).hex()
    assert one_shot == ref
    assert streamed == ref
    assert from_host == ref
    assert xof == oracle.keyed_hash_xof(data, key, 100).hex()
    assert default_mode == oracle.hash(data).hex()
    assert status == "0"

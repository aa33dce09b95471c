"""Build libb3g.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit is compiled by its own nvcc process (in parallel), then
linked into a shared library with the CUDA runtime linked statically, so that the
library loads on machines without a GPU driver (symbol checks) as well as on the GPU.

    python -m blake3_merkle_tree_gb300.build [--verbose-ptxas]
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libb3g.so")
SOURCES = ["b3g_leaf.cu", "b3g_reduce.cu", "b3g_api.cu", "b3g_noalloc.cu", "b3g_stream.cu"]
HEADERS = ["b3g_device.cuh", "b3g_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _flags(verbose_ptxas: bool) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-Xcompiler", "-Wall"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _inputs_newer_than(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "blake3_gb300.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile (if needed) and return the path of libb3g.so."""
    if not force and not verbose_ptxas and not _inputs_newer_than(LIB):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    flags = _flags(verbose_ptxas)

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc(), *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
        return obj, p.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="--verbose-ptxas" in sys.argv))

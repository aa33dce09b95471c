"""Resource guard for the leaf kernels (CPU: compiles only, no GPU).

The staged leaf kernels' throughput rests on five resident CTAs of 160 threads per SM,
which holds only while the register allocator stays at or below 80 registers per thread
(65,536 / (5 x 160) = 81.9, allocated in steps of 8).  The allocation moves with small
source changes (72, 95 and 113 registers have all been seen), so this test compiles the
leaf kernels with the package's own flags and reads ptxas's resource report.

- The bulk-tensor-copy kernel (leaf_tma_kernel) compiles to 72 registers without spill
  loads.
- The asynchronous-copy kernel (leaf_async_kernel) is held to five CTAs by its launch
  bounds and calls its reducer warp as a function (which calls its tree level in turn;
  the registers it keeps around that call are the called functions' own, not counted
  here).  The aligned kernels then spill nothing.  The misaligned ones (one more 16-byte
  unit and a shift per block) reload up to 28 bytes; the test caps them there.
"""
import os
import re
import shutil
import subprocess

import pytest

from blake3_merkle_tree_gb300 import build

# leaf_tma_kernel<C, S, LOAD, CHUNK_CVS, MODE> and leaf_async_kernel<C, S, CHUNK_CVS, MODE, MIS>
# as they appear in the mangled names
_TMA = re.compile(r"leaf_tma_kernelILi(\d+)ELi(\d+)ELi(\d+)ELb([01])ELj(\d+)E")
_ASYNC = re.compile(r"leaf_async_kernelILi(\d+)ELi(\d+)ELb([01])ELj(\d+)ELb([01])E")
_ASYNC_MAX_SPILL_LOADS_MISALIGNED = 28


def _ptxas_report(tmp_path, extra=()):
    nvcc = build.nvcc()
    if not (os.path.exists(nvcc) or shutil.which(nvcc)):
        pytest.skip("nvcc not available")
    obj = tmp_path / "leaf.o"
    cmd = [nvcc, *build._flags(True), *extra, "-c", os.path.join(build.CSRC, "b3g_leaf.cu"), "-o", str(obj)]
    p = subprocess.run(cmd, capture_output=True, text=True)
    assert p.returncode == 0, p.stderr[-4000:]
    kernels = {}
    cur, spills = None, None
    for line in p.stderr.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur, spills = m.group(1), None
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur:
            spills = (int(m.group(1)), int(m.group(2)))
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and cur:
            kernels[cur] = (int(m.group(1)), spills or (0, 0))
            cur = None
    return kernels


@pytest.mark.parametrize("staging", ["default", "tma"])
def test_leaf_kernels_keep_five_ctas_per_sm(tmp_path, staging):
    """The default build (asynchronous copies for every staged input) and the build with
    the bulk-tensor-copy staging for aligned inputs (B3G_STAGING=0), which stays buildable."""
    kernels = _ptxas_report(tmp_path, ["-DB3G_STAGING=0"] if staging == "tma" else [])
    tma = asy = 0
    for name, (regs, (_, spill_loads)) in kernels.items():
        m = _TMA.search(name)
        if m and int(m.group(1)) == 128:
            tma += 1
            what = "leaf_tma_kernel<{},{},{},{},{}>".format(*m.groups())
            assert regs <= 80, f"{what}: {regs} registers, five 160-thread CTAs per SM need at most 80"
            assert spill_loads == 0, f"{what}: {spill_loads} bytes of spill loads"
        m = _ASYNC.search(name)
        if m and int(m.group(1)) == 128:
            asy += 1
            what = "leaf_async_kernel<{},{},{},{},{}>".format(*m.groups())
            assert regs <= 80, f"{what}: {regs} registers, five 160-thread CTAs per SM need at most 80"
            limit = _ASYNC_MAX_SPILL_LOADS_MISALIGNED if m.group(5) == "1" else 0
            assert spill_loads <= limit, f"{what}: {spill_loads} bytes of spill loads"
    # one staging for aligned inputs (keyed and default mode, with and without the chunk-CV
    # output) and the asynchronous-copy kernel for misaligned ones (the same three)
    assert tma + asy == 6 and asy >= 3, sorted(kernels)
    assert tma == (3 if staging == "tma" else 0)

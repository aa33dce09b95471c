"""Resource guard for the leaf kernel (CPU: compiles only, no GPU).

The leaf kernel's throughput rests on five resident CTAs of 160 threads per SM, which
holds only while the register allocator stays at or below 80 registers per thread
(65,536 / (5 x 160) = 81.9, allocated in steps of 8), and on a hot loop without spill
loads.  The allocation moves with small source changes (72 and 95 registers have both
been seen), so this test compiles the leaf kernels with the package's own flags and
reads ptxas's resource report.
"""
import os
import re
import shutil
import subprocess

import pytest

from blake3_merkle_tree_gb300 import build

# leaf_tma_kernel<C, S, LOAD, CHUNK_CVS, MODE> as it appears in the mangled name
_NAME = re.compile(r"leaf_tma_kernelILi(\d+)ELi(\d+)ELi(\d+)ELb([01])ELj(\d+)E")


def _ptxas_report(tmp_path):
    nvcc = build.nvcc()
    if not (os.path.exists(nvcc) or shutil.which(nvcc)):
        pytest.skip("nvcc not available")
    obj = tmp_path / "leaf.o"
    cmd = [nvcc, *build._flags(True), "-c", os.path.join(build.CSRC, "b3g_leaf.cu"), "-o", str(obj)]
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


def test_leaf_kernel_keeps_five_ctas_per_sm(tmp_path):
    kernels = _ptxas_report(tmp_path)
    checked = 0
    for name, (regs, (_, spill_loads)) in kernels.items():
        m = _NAME.search(name)
        if not m or int(m.group(1)) != 128:
            continue
        checked += 1
        tile, stages, load, cvs, mode = (int(x) for x in m.groups())
        what = f"leaf_tma_kernel<{tile},{stages},{load},{cvs},{mode}>"
        assert regs <= 80, f"{what}: {regs} registers, five 160-thread CTAs per SM need at most 80"
        assert spill_loads == 0, f"{what}: {spill_loads} bytes of spill loads"
    # keyed and default mode, with and without the chunk-CV output
    assert checked == 3, sorted(kernels)

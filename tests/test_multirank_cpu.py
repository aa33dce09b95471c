"""The N > 1 host logic of bench.py on the CPU: two gloo ranks, and torchrun with two ranks.

With N ranks the digest is sharded (blake3_merkle_tree_gb300.sharded, tested with gloo
ranks in test_sharded_cpu.py); what the ranks share in the bench is the timing: a barrier
around the timed region, the maximum time over ranks, and the whole-job throughput over
all ranks' bytes.
"""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench._max_over_ranks(local_ms[rank], world, "cpu")
        value = bench._job_gbs(world * (1 << 30), 4, slowest)
        dist.barrier()
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    local_ms = [12.5, 20.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, slowest, value in results:
        assert slowest == 20.0  # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * (1 << 30) * 4 / 0.020 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench._max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench._job_gbs(10 ** 9, 2, 1000.0) == pytest.approx(2.0)


def test_launch_and_work_counts():
    sys.path.insert(0, ROOT)
    import bench

    # reduction launches: groups of 64 CVs up to 32,768, else 1024
    assert [bench._reduce_launches(c) for c in (1, 32, 64, 65, 2048, 32768, 32769, 98305)] == \
        [0, 1, 1, 2, 2, 3, 2, 2]
    # 12 GiB + 777: 16 per full chunk, 13 blocks of the 777-byte chunk, parents inside tiles
    n = 12 * (1 << 30) + 777
    assert bench._leaf_compressions(n, 98305) == 12582912 * 16 + 13 + (12582913 - 98305)
    assert bench._leaf_compressions(1 << 20, 8) == 1024 * 16 + 1024 - 8


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`bench.py --impl reference` is the CPU oracle: under torchrun only rank 0 runs it."""
    env = dict(os.environ, B3G_REF_BUDGET_S="2", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"

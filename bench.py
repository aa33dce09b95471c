#!/usr/bin/env python3
"""Throughput of the keyed BLAKE3 digest of one buffer resident in GPU memory.

One step = one pass of the whole path over the 12 GiB + 777 byte workload
(uniform bytes, data seed 6, key seed 7): the leaf kernel (chunk compression fused
with the CTA subtree) followed by the reduction of the CTA roots to the ROOT digest.
The input (12.9 GB) is far larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is GB/s hashed (10^9 bytes of input per second) with
the input already in HBM; `e2e` is the same metric through the public C-ABI call
with the input copied from pinned host memory every step and the digest read back;
`roofline` relates the leaf kernel (the dominant one) to the integer-issue peak of
the GPU; `cpu_baseline` times the CPU oracle on a bounded prefix of the workload.
`--impl reference` times the CPU oracle alone as the reference arm.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

from blake3_merkle_tree_gb300 import workloads  # noqa: E402

METRIC = "GB/s hashed (keyed BLAKE3, 1 GB300)"
WORKLOAD = "12GiB+777"
# Integer work of one compression under the plain instruction count: 7 rounds x 8 G
# x 12 operations (6 adds with the two 3-input adds fused, 4 XORs, 4 rotates ->
# 2 IADD3 + 2 IADD + 4 XOR + 4 rotates) + 8 XORs for the output CV.
OPS_PER_COMPRESSION = 7 * 8 * 12 + 8
# The page's count: 6 operations per G, 336 per 64-byte block ("BLAKE3 GPU 400x faster hashing",
# section "压缩函数").
PAGE_OPS_PER_COMPRESSION = 336
DYNAMIC_MIN_TILES = 760  # above this many CTA subtrees the leaf kernel takes tiles from a counter
INT32_LANES_PER_SM = 128  # integer instructions issued per SM per clock (4 schedulers x 32 lanes)


def _peaks():
    p = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region (read through a pipe)."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.reader = None

    def __enter__(self):
        import threading

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.reader = threading.Thread(target=lambda: self.lines.extend(self.proc.stdout), daemon=True)
        self.reader.start()
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=5)

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in list(self.lines):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            if self.gpu and self.gpu.lower() not in parts[0].lower():
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 0.5 * max(x[2] for x in rows)] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in loaded for n, v in zip(names, r[3][1:]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(loaded), "reasons": reasons}


def _leaf_sources_sha256() -> str:
    """SHA-256 (first 16 hex digits) of the sources the leaf kernels are built from: a
    counter capture holds for the kernel only while these are unchanged."""
    import hashlib

    csrc = os.path.join(HERE, "blake3_merkle_tree_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("b3g_leaf.cu", "b3g_device.cuh", "b3g_internal.h"):
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_per_launch(lib, nchunks):
    """DRAM bytes and issued thread instructions of one leaf launch, scaled by chunks from
    the ncu capture recorded in profiles/leaf_*_traffic.json for the kernel configuration
    built and the leaf sources as they are; None if there is none (the kernel changed
    since the counters were taken)."""
    cfg = lib.blake3_kernel_config().decode()
    src = _leaf_sources_sha256()
    rec = None
    for name in ("leaf_async_kernel_traffic.json", "leaf_tma_kernel_traffic.json"):
        p = os.path.join(HERE, "profiles", name)
        if os.path.exists(p):
            with open(p) as f:
                r = json.load(f)
            if r.get("kernel_config") == cfg and r.get("leaf_sources_sha256") == src:
                rec = r
                break
    if rec is None:
        return None, "no capture of this kernel configuration and these leaf sources", None
    per_chunk = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) / rec["chunks"]
    issued = None
    if "warp_inst_executed" in rec:
        issued = rec["warp_inst_executed"] * 32 / rec["chunks"] * nchunks
    return (per_chunk * nchunks, f"ncu capture on {rec['workload']} scaled by chunks ({rec['chunks']} -> {nchunks})",
            issued)


def _max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks: a job takes as long as its slowest rank."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _job_gbs(job_bytes: int, steps: int, total_ms: float) -> float:
    """Whole-job GB/s: the bytes all ranks hash per step, over the slowest rank's time."""
    return job_bytes * steps / (total_ms / 1e3) / 1e9


def _reduce_launches(count: int) -> int:
    """Launches of the root reduction of `count` CVs (groups of 64 up to 32,768 CVs, else 1024)."""
    group = 64 if count <= 32768 else 1024
    launches = 0
    while count > 1:
        count = -(-count // group)
        launches += 1
    return launches


def _leaf_compressions(nbytes: int, tiles: int) -> int:
    """Compressions of the leaf kernel over `nbytes` in `tiles` 128-chunk subtrees: 16 per
    full chunk, one per block of the partial chunk, and the parents inside the subtrees."""
    nchunks = max(1, -(-nbytes // 1024))
    tail = nbytes % 1024
    return (nbytes // 1024) * 16 + ((tail + 63) // 64 if tail else 0) + (nchunks - tiles)


def _sources_sha256() -> str:
    """SHA-256 of the library's CUDA/C sources and the C header (first 16 hex digits): the
    identity of the measured build, also where no version-control metadata travels."""
    import hashlib

    root = os.path.dirname(os.path.abspath(__file__))
    csrc = os.path.join(root, "blake3_merkle_tree_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    files.append(os.path.join(root, "include", "blake3_gb300.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _oracle_sample(host_bytes: torch.Tensor, key: bytes, target_s: float):
    """Time the CPU oracle on doubling prefixes until one run takes >= target_s."""
    import oracle

    n = min(64 << 20, host_bytes.numel())
    while True:
        t0 = time.perf_counter()
        oracle.keyed_hash(host_bytes[:n], key)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= host_bytes.numel():
            return n, dt
        n = min(host_bytes.numel(), n * max(2, int(target_s / max(dt, 1e-3) * 0.9)))


def _oracle_threaded(host_bytes: torch.Tensor, key: bytes, threads: int):
    """All host cores through the unchanged oracle functions: the largest power-of-two
    prefix of whole chunks is split into equal aligned subtrees, hashed by parallel
    threads (the ctypes calls release the GIL), and folded pairwise on one thread with
    ROOT on the top parent.  Checked against the plain oracle on a small prefix first."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    def digest(data, t):
        chunks = data.numel() // 1024
        per = chunks // t
        with ThreadPoolExecutor(t) as ex:
            cvs = list(ex.map(lambda i: oracle.subtree_cv(data[i * per * 1024:(i + 1) * per * 1024], key, i * per),
                              range(t)))
        while len(cvs) > 1:
            cvs = [oracle.parent_cv(key, cvs[2 * j], cvs[2 * j + 1], len(cvs) == 2) for j in range(len(cvs) // 2)]
        return cvs[0]

    chunks = host_bytes.numel() // 1024
    if chunks < 2 * threads:
        return None
    p2 = 1 << (chunks.bit_length() - 1)
    t = 1 << (threads.bit_length() - 1)
    check = host_bytes[:min(p2, 1 << 14) * 1024]
    if digest(check, t) != oracle.keyed_hash(check, key):
        raise RuntimeError("threaded oracle fold differs from the oracle")
    data = host_bytes[:p2 * 1024]
    t0 = time.perf_counter()
    digest(data, t)
    dt = time.perf_counter() - t0
    return {"value": p2 * 1024 / dt / 1e9, "unit": "GB/s", "cores": t, "kind": "oracle, one thread per aligned subtree",
            "sample": f"first {p2 * 1024} bytes of the workload as one input: {t} subtrees of {p2 // t} chunks "
                      f"hashed in parallel by the unchanged oracle, folded on one thread ({dt:.1f} s)"}


def _oracle_digest_threaded(host_bytes: torch.Tensor, key: bytes, threads: int) -> bytes:
    """The oracle's digest of the whole input on all host cores: the tree is split the
    way the specification splits it (left subtree = the largest power of two of chunks
    below the count) until every piece holds at most 1/threads of the chunks; the pieces
    are hashed in parallel by the unchanged oracle (oracle.subtree_cv, the ctypes call
    releases the GIL), and the parents above them are folded on one thread with ROOT on
    the top one."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    n = host_bytes.numel()
    nchunks = max(1, -(-n // 1024))
    if nchunks == 1 or threads <= 1:
        return oracle.keyed_hash(host_bytes, key)
    per = max(1, -(-nchunks // threads))
    leaves = []  # (first chunk, chunk count), left to right

    def split(lo, cnt):
        if cnt <= per:
            leaves.append((lo, cnt))
            return
        left = 1 << ((cnt - 1).bit_length() - 1)
        split(lo, left)
        split(lo + left, cnt - left)

    split(0, nchunks)
    with ThreadPoolExecutor(threads) as ex:
        cvs = dict(zip(leaves, ex.map(
            lambda lc: oracle.subtree_cv(host_bytes[lc[0] * 1024:min(n, (lc[0] + lc[1]) * 1024)], key, lc[0]),
            leaves)))

    def fold(lo, cnt, root):
        if (lo, cnt) in cvs:
            return cvs[(lo, cnt)]
        left = 1 << ((cnt - 1).bit_length() - 1)
        return oracle.parent_cv(key, fold(lo, left, False), fold(lo + left, cnt - left, False), root)

    return fold(0, nchunks, True)


def _host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def _step_fn(lib, binding, dev, n, key, stream):
    """One pass of the path over `dev`: the leaf launch (chunk CVs and CTA subtrees), then
    the reduction launches to the ROOT digest.  The leaf kernel's tile counter is zeroed
    once here: every launch that completes leaves it zero.  Returns (step, digest tensor,
    launches, tiles)."""
    sp = stream.cuda_stream
    leaves_log2 = -1
    tiles = lib.blake3_tile_count(n, leaves_log2)
    roots = torch.empty((tiles, 32), dtype=torch.uint8, device="cuda")
    red_ws = torch.empty(max(16, lib.blake3_reduce_workspace_size(tiles, -1)), dtype=torch.uint8, device="cuda")
    out = torch.empty(32, dtype=torch.uint8, device="cuda")
    counter = torch.zeros(4, dtype=torch.int32, device="cuda")  # the leaf kernel's tile counter

    # as in the library's one-shot call: the counter only when there are more tiles than
    # resident CTAs (below that every CTA has one tile)
    dynamic = tiles > DYNAMIC_MIN_TILES

    def step(ev_a=None, ev_b=None):
        if ev_a is not None:
            ev_a.record(stream)
        st = lib.blake3_keyed_tile_roots_ex(dev.data_ptr(), n, 0, key, leaves_log2, 1, roots.data_ptr(),
                                            counter.data_ptr() if dynamic else None, sp)
        if st:
            raise binding.B3GError(st, "blake3_keyed_tile_roots")
        if ev_b is not None:
            ev_b.record(stream)
        if tiles > 1:
            st = lib.blake3_keyed_reduce_cvs(roots.data_ptr(), tiles, key, 1, -1, out.data_ptr(), red_ws.data_ptr(),
                                             red_ws.numel(), sp)
            if st:
                raise binding.B3GError(st, "blake3_keyed_reduce_cvs")

    return step, (roots[0] if tiles == 1 else out), 1 + _reduce_launches(tiles), tiles


def _roofline_fracs(n, tiles, leaf_s, hbm_peak, int_peak):
    """The fractions of one leaf launch over n bytes: against the min roofline
    (min(HBM peak, INT32 issue peak / the page's ops per byte), which is the HBM peak on
    GB300), and against the issue peak with the plain instruction count."""
    comps = _leaf_compressions(n, tiles)
    page_bound = min(hbm_peak, int_peak / (comps * PAGE_OPS_PER_COMPRESSION / n) / 1e9)
    gbs = n / leaf_s / 1e9
    return {"leaf_GBps": gbs, "frac_of_min_roofline": gbs / page_bound, "min_roofline_GBps": page_bound,
            "frac_hbm": gbs / hbm_peak,
            "frac_issue_bound": comps * OPS_PER_COMPRESSION / leaf_s / int_peak}


def _measure_config(lib, binding, wname, steps, hbm_peak, int_peak, threads):
    """One configuration of the benchmark: GB/s of the leaf + reduction step, the roofline
    fractions of the leaf launch, and the digest against the oracle (on all host cores).

    An input that fits in the L2 is timed step by step (median of per-step CUDA events),
    with the L2 flushed before each step.  A larger one is timed as K steps back to back
    between two events, as the headline is: an event recorded between two launches ends
    the early launch of the second (programmatic dependent launch), which costs a few
    microseconds per step.  The leaf launch's own time comes from per-step events in
    both cases."""
    w = workloads.WORKLOADS[wname]
    key = w.key()
    n = w.nbytes
    dev = w.data(device="cuda")
    stream = torch.cuda.current_stream()
    step, digest_t, launches, tiles = _step_fn(lib, binding, dev, n, key, stream)
    small = n < (256 << 20)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if small else None
    for _ in range(3):
        step()
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(steps)]
    for z, a, b, c in evs:
        if flush is not None:
            flush.fill_(1)
        z.record(stream)
        step(a, b)
        c.record(stream)
    torch.cuda.synchronize()
    step_ms_events = statistics.median(z.elapsed_time(c) for z, _, _, c in evs)
    leaf_ms = statistics.median(a.elapsed_time(b) for _, a, b, _ in evs)
    step_ms = step_ms_events
    if not small:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        step_ms = e0.elapsed_time(e1) / steps
    got = bytes(digest_t.cpu().numpy())
    t0 = time.perf_counter()
    ref = _oracle_digest_threaded(dev.cpu(), key, threads)
    oracle_s = time.perf_counter() - t0
    res = {"workload": f"{w.name} keyed BLAKE3, {w.kind} bytes seed {w.data_seed}, key seed {w.key_seed}",
           "bytes": n, "steps": steps, "GBps": n / step_ms / 1e6, "ms_per_step": step_ms, "leaf_ms": leaf_ms,
           "gpu_launches_per_step": launches,
           "timing": "median of per-step events" if small else f"{steps} steps back to back between two events",
           "GBps_per_step_events": n / step_ms_events / 1e6,
           "l2": "flushed between steps (256 MiB write)" if small else "input larger than L2",
           "digest": got.hex(), "digest_equals_oracle": got == ref,
           "oracle": f"unchanged oracle on {threads} host threads, {oracle_s:.1f} s"}
    res.update(_roofline_fracs(n, tiles, leaf_ms / 1e3, hbm_peak, int_peak))
    if not small:
        res["l2_flush_needed"] = False
    del dev, flush
    torch.cuda.empty_cache()
    return res


def _ragged_config(binding):
    """The ragged-length sweep (13 fixed and 64 seeded lengths): every digest through the
    public call against the oracle."""
    import oracle

    lengths = workloads.ragged_lengths()
    key = workloads.key_bytes(workloads.RAGGED_KEY_SEED)
    bad = []
    for length in lengths:
        host = workloads.uniform_bytes(length, length)
        got = bytes(binding.blake3_keyed_hash(host.to("cuda"), key).cpu().numpy())
        if got != oracle.keyed_hash(host, key):
            bad.append(length)
    return {"workload": "ragged-length sweep: 13 fixed + 64 seeded lengths in [1, 4 MiB], seed = length, key seed 1",
            "lengths": len(lengths), "digests_equal_oracle": len(lengths) - len(bad), "mismatched_lengths": bad}


def run_reference(args):
    """Reference arm: the CPU oracle, timed on the host cores, on bounded prefixes."""
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle

    w = workloads.WORKLOADS[WORKLOAD]
    key = w.key()
    # size the per-step sample so that warm-up + timed steps take about a minute
    probe = workloads.uniform_bytes(w.data_seed, 16 << 20)
    t0 = time.perf_counter()
    oracle.keyed_hash(probe, key)
    speed = probe.numel() / (time.perf_counter() - t0)
    budget_s = float(os.environ.get("B3G_REF_BUDGET_S", "60"))
    sample = int(speed * budget_s / (args.steps + args.warmup))
    sample = max(1 << 20, min(w.nbytes, sample - sample % 1024))
    host = workloads.uniform_bytes(w.data_seed, sample)
    for _ in range(args.warmup):
        oracle.keyed_hash(host, key)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.keyed_hash(host, key)
    dt = time.perf_counter() - t0
    value = args.steps * sample / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} keyed BLAKE3, uniform bytes seed 6, key seed 7",
                   "bytes": w.nbytes, "sample_bytes_per_step": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu_model": _cpu_model(),
                         "sample": f"first {sample} bytes of the workload, hashed as a whole input, per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    from blake3_merkle_tree_gb300 import binding, build

    world, rank, local = _dist()
    if world > 1:
        return run_sharded(args, world, rank, local)
    torch.cuda.set_device(local)
    build.build()
    lib = binding.library()

    w = workloads.WORKLOADS[args.workload]
    key = w.key()
    n = w.nbytes
    dev = w.data(device="cuda")
    stream = torch.cuda.current_stream()
    leaves_log2 = lib.blake3_default_leaves_log2()
    # per step: the tile counter zeroed, the leaf launch (timed alone as well), the
    # reduction launches
    step, digest_t, launches, tiles = _step_fn(lib, binding, dev, n, key, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    digest_bench = bytes(digest_t.cpu().numpy())
    digest_api = bytes(binding.blake3_keyed_hash(dev, key).cpu().numpy())
    if digest_bench != digest_api:
        raise RuntimeError("bench step and blake3_keyed_hash disagree")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    gpu_id = str(getattr(props, "uuid", "") or "")
    with ClockSampler(gpu_id) as clk:
        for i in range(args.steps):
            step(starts[i], mids[i])
        end.record(stream)
        torch.cuda.synchronize()
    total_ms = starts[0].elapsed_time(end)
    leaf_ms = [starts[i].elapsed_time(mids[i]) for i in range(args.steps)]
    step_ms = [starts[i].elapsed_time(starts[i + 1] if i + 1 < args.steps else end) for i in range(args.steps)]
    timing = {"step_ms_median": statistics.median(step_ms), "step_ms_min": min(step_ms),
              "leaf_ms_median": statistics.median(leaf_ms),
              "reduction_and_gaps_ms_median": statistics.median(s - l for s, l in zip(step_ms, leaf_ms))}
    ms_per_step = total_ms / args.steps
    value = _job_gbs(n, args.steps, total_ms)

    # roofline of the leaf kernel (integer issue bound)
    nchunks = max(1, -(-n // 1024))
    nfull = n // 1024
    tail = n % 1024
    leaf_compressions = _leaf_compressions(n, tiles)
    ops = leaf_compressions * OPS_PER_COMPRESSION
    page_ops = leaf_compressions * PAGE_OPS_PER_COMPRESSION
    leaf_s = statistics.mean(leaf_ms) / 1e3
    peaks, peak_kind = _peaks()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    clocks = clk.summary()
    peak_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    int_peak = sms * INT32_LANES_PER_SM * peak_mhz * 1e6  # ops/s
    achieved = ops / leaf_s
    roofline = {
        "bound": "alu", "achieved": achieved / 1e9, "peak": int_peak / 1e9, "unit": "Gop/s",
        "frac": achieved / int_peak, "traffic": None,
        "ops_per_launch": ops, "ops_per_byte": ops / n, "leaf_ms": statistics.mean(leaf_ms),
        "peak_basis": f"{sms} SMs x {INT32_LANES_PER_SM} int32 lanes x {peak_mhz:.0f} MHz (derived)",
        "page_count": {"ops_per_byte": page_ops / n, "achieved": page_ops / leaf_s / 1e9,
                       "frac": page_ops / leaf_s / int_peak},
        "hbm": {"achieved": n / leaf_s / 1e9, "peak": float(peaks.get("hbm_gbs", 6800.0)), "unit": "GB/s",
                "frac": n / leaf_s / 1e9 / float(peaks.get("hbm_gbs", 6800.0)), "peak_kind": peak_kind},
        "issue_bound_GBps": int_peak / (ops / n) / 1e9,
    }
    # the min roofline: the slower of the input bytes at the HBM peak and the page's
    # integer operations per byte at the INT32 issue peak (the HBM peak on GB300)
    fr = _roofline_fracs(n, tiles, leaf_s, float(peaks.get("hbm_gbs", 6800.0)), int_peak)
    roofline["roofline_gbs"] = fr["min_roofline_GBps"]
    roofline["frac_of_min_roofline"] = fr["frac_of_min_roofline"]
    roofline["frac_issue_bound"] = fr["frac_issue_bound"]
    roofline["definitions"] = {
        "frac": "680 integer instructions per compression (the plain count) / the INT32 issue peak",
        "frac_of_min_roofline": "input bytes / min(HBM peak, INT32 issue peak / the page's 336 ops per block) "
                                "(the HBM peak on this GPU)",
        "frac_issue_bound": "same as frac"}
    traffic, traffic_src, issued = _traffic_per_launch(lib, nchunks)
    roofline["traffic"] = traffic
    roofline["traffic_source"] = traffic_src
    if issued is not None:
        # the same peak against the instructions the kernel actually issues (ncu inst_executed)
        roofline["issued"] = {"instructions_per_byte": issued / n, "achieved": issued / leaf_s / 1e9,
                              "frac": issued / leaf_s / int_peak, "unit": "G instructions/s"}
    roofline["algorithmic_bytes"] = n
    roofline["kernel_config"] = lib.blake3_kernel_config().decode()

    # end to end through the public call, host buffers, copies inside the timed region
    e2e = None
    host = None
    if not args.no_e2e:
        e2e, host = _e2e(args, binding, dev, key, digest_api)

    cpu = None
    if not args.no_cpu_baseline:
        if host is None:
            host = dev.cpu()
        sample, dt = _oracle_sample(host, key, args.cpu_seconds)
        cpu = {"value": sample / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu_model": _cpu_model(),
               "sample": f"first {sample} bytes of the workload hashed as one input by the single-threaded "
                         f"C oracle ({dt:.1f} s)"}
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        if cores > 1:
            cpu["all_cores"] = _oracle_threaded(host, key, cores)

    # the headline digest against the oracle, on all host cores
    digest_oracle = None
    if not args.no_oracle_check:
        if host is None:
            host = dev.cpu()
        t0 = time.perf_counter()
        ok = _oracle_digest_threaded(host, key, _host_cores()) == digest_api
        digest_oracle = {"equal": ok, "threads": _host_cores(), "seconds": round(time.perf_counter() - t0, 1)}
    del host

    # the other configurations of the workload set, each with its own GB/s, roofline
    # fractions and oracle check (C5, the largest, is the headline above)
    configs = None
    if not args.no_configs:
        hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
        th = _host_cores()
        configs = {
            "C1_1MiB": _measure_config(lib, binding, "1MiB", 200, hbm_peak, int_peak, th),
            "C2_ragged": _ragged_config(binding),
            "C3_bf16_256MiB": _measure_config(lib, binding, "bf16_256MiB", 50, hbm_peak, int_peak, th),
            "C4_4GiB": _measure_config(lib, binding, "4GiB", 20, hbm_peak, int_peak, th),
        }
        configs["C4_4GiB"]["target"] = "frac_issue_bound >= 0.70 (at least 70 % of the roofline for inputs of 4 GiB and more)"

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": f"{w.name} keyed BLAKE3, {w.kind} bytes seed {w.data_seed}, key seed {w.key_seed}",
                   "input": "u8 bytes, hashed as little-endian u32 words", "bytes": n, "chunks": nchunks,
                   "leaves_per_cta": 1 << leaves_log2, "cta_roots": tiles,
                   "l2": f"input {n / 1e9:.2f} GB > 126 MB L2; no flush needed", "parallelism": "one GPU",
                   "sources_sha256": _sources_sha256()},
        "timing": timing, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches * args.steps, "clocks": clocks,
        "digest": digest_api.hex(), "digest_vs_oracle": digest_oracle, "configs": configs,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_sharded(args, world, rank, local):
    """N > 1: one buffer of N times the workload's length (bytes [0, N * len) of the same
    seeded stream), sharded over the ranks in 128-chunk tiles, so every GPU holds the
    workload's length give or take one tile (weak scaling).  A step is the leaf launch on
    the rank's slice, an all-gather of the tile roots over NCCL and the fold to the ROOT
    digest on every rank (blake3_merkle_tree_gb300.sharded)."""
    import torch.distributed as dist
    from blake3_merkle_tree_gb300 import binding, build, sharded

    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    lib = binding.library()
    w = workloads.WORKLOADS[args.workload]
    if w.kind != "uniform":
        raise SystemExit(f"{w.name}: the sharded run needs a uniform workload")
    key = w.key()
    total = world * w.nbytes
    sd = sharded.ShardedDigest(total, key)
    n_loc = sd.end - sd.start
    n_tiles = sd.t1 - sd.t0
    dev = w.data_range(sd.start, n_loc, device="cuda")
    stream = torch.cuda.current_stream()

    for _ in range(max(3, args.warmup)):
        sd(dev)
    torch.cuda.synchronize()
    digest = bytes(sd.out.cpu().numpy())
    mine = torch.tensor(list(digest), dtype=torch.uint8, device="cuda")
    every = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(every, mine)
    if any(bytes(x.cpu().numpy()) != digest for x in every):
        raise RuntimeError("the ranks disagree on the sharded digest")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    end = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    gpu_id = str(getattr(props, "uuid", "") or "")
    with ClockSampler(gpu_id) as clk:
        for i in range(args.steps):
            starts[i].record(stream)
            sd(dev, after_leaf=lambda e=mids[i]: e.record(stream))
        end.record(stream)
        torch.cuda.synchronize()
    dist.barrier()
    total_ms = _max_over_ranks(starts[0].elapsed_time(end), world, "cuda")
    leaf_ms = [starts[i].elapsed_time(mids[i]) for i in range(args.steps)]
    step_ms = [starts[i].elapsed_time(starts[i + 1] if i + 1 < args.steps else end) for i in range(args.steps)]
    timing = {"step_ms_median": statistics.median(step_ms), "step_ms_min": min(step_ms),
              "leaf_ms_median": statistics.median(leaf_ms),
              "gather_and_fold_ms_median": statistics.median(x - y for x, y in zip(step_ms, leaf_ms)),
              "note": "this rank's (rank 0's) events; the value uses the slowest rank's total"}
    value = _job_gbs(total, args.steps, total_ms)

    # roofline of this rank's leaf launch (integer issue bound)
    peaks, peak_kind = _peaks()
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    peak_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    int_peak = sms * INT32_LANES_PER_SM * peak_mhz * 1e6
    leaf_s = statistics.mean(leaf_ms) / 1e3
    ops = _leaf_compressions(n_loc, n_tiles) * OPS_PER_COMPRESSION
    nchunks = max(1, -(-n_loc // 1024))
    traffic, traffic_src, _ = _traffic_per_launch(lib, nchunks)
    roofline = {"bound": "alu", "achieved": ops / leaf_s / 1e9, "peak": int_peak / 1e9, "unit": "Gop/s",
                "frac": ops / leaf_s / int_peak, "traffic": traffic, "traffic_source": traffic_src,
                "ops_per_launch": ops, "leaf_ms": statistics.mean(leaf_ms), "algorithmic_bytes": n_loc,
                "peak_basis": f"{sms} SMs x {INT32_LANES_PER_SM} int32 lanes x {peak_mhz:.0f} MHz (derived)",
                "peak_kind": peak_kind, "kernel_config": lib.blake3_kernel_config().decode()}

    # end to end: each rank's slice from pinned host memory, copies overlapped with the
    # leaf launches, then the gather, the fold and the 32-byte digest back to the host
    e2e = None
    if not args.no_e2e:
        host = torch.empty(n_loc, dtype=torch.uint8, pin_memory=True)
        host.copy_(dev)
        sd.from_host(host)
        torch.cuda.synchronize()
        dist.barrier()
        step_s = []
        for _ in range(max(1, min(args.e2e_steps, args.steps))):
            t0 = time.perf_counter()
            got = bytes(sd.from_host(host).cpu().numpy())
            step_s.append(time.perf_counter() - t0)
            if got != digest:
                raise RuntimeError("end-to-end sharded digest differs")
        e2e_s = _max_over_ranks(statistics.median(step_s), world, "cuda")
        e2e = {"value": total / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": total,
               "d2h_bytes_per_step": 32 * world, "ms_per_step": e2e_s * 1e3, "steps": len(step_s),
               "ms_each_step": [round(x * 1e3, 2) for x in step_s], "statistic": "median step, slowest rank",
               "call": "ShardedDigest.from_host (pinned host slice per rank, 2 x 256 MiB device slots)"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": f"{world} x {w.name} keyed BLAKE3 as one buffer, {w.kind} bytes seed {w.data_seed}, "
                               f"key seed {w.key_seed}",
                   "input": "u8 bytes, hashed as little-endian u32 words", "bytes": total,
                   "bytes_this_rank": n_loc, "tiles": sd.tiles, "tiles_this_rank": n_tiles,
                   "l2": f"input {n_loc / 1e9:.2f} GB per GPU > 126 MB L2; no flush needed",
                   "parallelism": f"sharded{world}",
                   "exchange": "all-gather of the 32-byte tile roots over NCCL, fold on every rank",
                   "sources_sha256": _sources_sha256()},
        "timing": timing, "roofline": roofline, "cpu_baseline": None, "e2e": e2e,
        "gpu_launches": (int(n_tiles > 0) + _reduce_launches(sd.tiles)) * args.steps,
        "clocks": clk.summary(), "digest": digest.hex(),
    }
    dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def _h2d_link_gbs(dev, host, warm=True):
    """The host->device link alone: the pinned buffer copied in 256 MiB pieces on one
    stream (one copy of the whole buffer runs far slower)."""
    n = dev.numel()
    piece = 256 << 20
    if warm:
        for a in range(0, min(n, 4 * piece), piece):
            dev[a:a + piece].copy_(host[a:a + piece], non_blocking=True)
    torch.cuda.synchronize()
    c0 = time.perf_counter()
    for a in range(0, n, piece):
        dev[a:a + piece].copy_(host[a:a + piece], non_blocking=True)
    torch.cuda.synchronize()
    return n / (time.perf_counter() - c0) / 1e9


def _e2e(args, binding, dev, key, digest_api):
    """The digest of the workload from pinned host memory through blake3_keyed_hash_host:
    every step copies the whole input host->device (overlapped with hashing inside the
    call) and returns the 32-byte digest to the host.  Each step is timed on its own and
    the value is taken from the median step (the host link is shared with other jobs on
    the machine); the link alone is measured before and after for context."""
    n = dev.numel()
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    host.copy_(dev)
    staging = torch.empty(3328 + 2 * (256 << 20), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    link_before = _h2d_link_gbs(dev, host)
    got = binding.blake3_keyed_hash_host(host, key, staging)  # warm-up
    step_s, link_each = [], []
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        got = binding.blake3_keyed_hash_host(host, key, staging)
        step_s.append(time.perf_counter() - t0)
        if got != digest_api:
            raise RuntimeError("end-to-end digest differs")
        link_each.append(_h2d_link_gbs(dev, host, warm=False))  # the link alone, right after
    e2e_s = statistics.median(step_s)
    link_after = _h2d_link_gbs(dev, host)
    e2e = {"value": n / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": n,
           "d2h_bytes_per_step": 32, "ms_per_step": e2e_s * 1e3, "steps": e2e_steps,
           "ms_each_step": [round(x * 1e3, 2) for x in step_s], "statistic": "median step",
           "h2d_copy_GBps_after_each_step": [round(x, 1) for x in link_each],
           "call": "blake3_keyed_hash_host (pinned host input, 2 x 256 MiB device staging)",
           "h2d_copy_GBps_before": link_before, "h2d_copy_GBps_after": link_after}
    return e2e, host


def _timed(fn, steps, warmup):
    """Mean milliseconds of fn() over `steps` calls after `warmup`, CUDA events on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_mode(args):
    """Measurements of the extensions, one JSON line each (not the headline)."""
    from blake3_merkle_tree_gb300 import binding, build

    torch.cuda.set_device(0)
    build.build()
    binding.library()
    if args.mode == "xof":
        w = workloads.WORKLOADS["1MiB"]
        d = w.data(device="cuda")
        out_len = args.xof_bytes
        out = torch.empty(out_len, dtype=torch.uint8, device="cuda")
        ms = _timed(lambda: binding.blake3_keyed_hash_xof(d, w.key(), out_len, out=out), args.steps, args.warmup)
        line = {"mode": "xof", "metric": "GB/s of extendable output (keyed BLAKE3, 1 GB300)",
                "value": out_len / ms / 1e6, "unit": "GB/s", "ms_per_call": ms,
                "config": {"input": "1MiB uniform seed 0, key seed 1", "out_bytes": out_len},
                "ops_per_output_byte": OPS_PER_COMPRESSION / 64}
    elif args.mode == "stream":
        w = workloads.WORKLOADS[args.workload]
        d = w.data(device="cuda")
        seg = args.segment_bytes
        h = binding.Hasher(w.key())
        segs = [d[a:a + seg] for a in range(0, d.numel(), seg)]

        def run():
            h.reset()
            for t in segs:
                h.update(t)
            h.finalize(out=out32)

        def run_many():
            h.reset()
            h.update_many(segs)
            h.finalize(out=out32)

        out32 = torch.empty(32, dtype=torch.uint8, device="cuda")
        one = bytes(binding.blake3_keyed_hash(d, w.key()).cpu().numpy())
        ms = _timed(run, args.steps, args.warmup)
        if bytes(out32.cpu().numpy()) != one:
            raise RuntimeError("streaming digest differs from the one-shot digest")
        ms_many = _timed(run_many, args.steps, args.warmup)
        if bytes(out32.cpu().numpy()) != one:
            raise RuntimeError("update_many digest differs from the one-shot digest")
        # the same C-ABI call with its pointer and length arrays built once, outside the
        # timed region: the library's cost without Python's per-segment marshalling
        lib = binding.library()
        ptrs = (ctypes.c_void_p * len(segs))(*[t.data_ptr() for t in segs])
        lens = (ctypes.c_uint64 * len(segs))(*[t.numel() * t.element_size() for t in segs])
        cur = torch.cuda.current_stream().cuda_stream

        def run_many_c():
            h.reset()
            if lib.blake3_hasher_update_many(h._h, ptrs, lens, len(segs), cur) != 0:
                raise RuntimeError("blake3_hasher_update_many failed")
            h.finalize(out=out32)

        ms_many_c = _timed(run_many_c, args.steps, args.warmup)
        if bytes(out32.cpu().numpy()) != one:
            raise RuntimeError("update_many (C arrays) digest differs from the one-shot digest")
        ms_one = _timed(lambda: binding.blake3_keyed_hash(d, w.key(), out=out32), args.steps, args.warmup)
        line = {"mode": "stream", "metric": "GB/s hashed through the streaming hasher (keyed BLAKE3, 1 GB300)",
                "value": d.numel() / ms / 1e6, "unit": "GB/s", "ms_per_digest": ms,
                "update_many_GBps": d.numel() / ms_many / 1e6,
                "update_many_prebuilt_arrays_GBps": d.numel() / ms_many_c / 1e6,
                "one_shot_GBps": d.numel() / ms_one / 1e6,
                "config": {"workload": w.name, "segment_bytes": seg, "segments": -(-d.numel() // seg)}}
    elif args.mode == "default":
        # the default (unkeyed) mode on the same workload, through the public one-shot
        # call, beside the keyed call
        w = workloads.WORKLOADS[args.workload]
        d = w.data(device="cuda")
        out32 = torch.empty(32, dtype=torch.uint8, device="cuda")
        ws = torch.empty(max(16, binding.blake3_workspace_size(d.numel())), dtype=torch.uint8, device="cuda")
        ms = _timed(lambda: binding.blake3_hash_ws(d, ws, out=out32), args.steps, args.warmup)
        ms_keyed = _timed(lambda: binding.blake3_keyed_hash_ws(d, w.key(), ws, out=out32), args.steps, args.warmup)
        line = {"mode": "default", "metric": "GB/s hashed in the default (unkeyed) mode (BLAKE3, 1 GB300)",
                "value": d.numel() / ms / 1e6, "unit": "GB/s", "ms_per_digest": ms,
                "keyed_GBps": d.numel() / ms_keyed / 1e6,
                "config": {"workload": w.name, "call": "blake3_hash_ws / blake3_keyed_hash_ws"}}
    elif args.mode == "ceiling":
        # the compression alone (messages in registers, no loads, no tree): the ceiling the
        # leaf kernel runs against, at its own 20 consumer warps per SM and at 32
        props = torch.cuda.get_device_properties(0)
        sms = props.multi_processor_count
        sink = torch.zeros(1, dtype=torch.int32, device="cuda")
        iters = 256
        rates = {}
        for warps in (20, 32):
            blocks = sms * warps // 4
            ms = _timed(lambda b=blocks: binding.blake3_selftest_compress_rate(b, iters, sink), args.steps,
                        args.warmup)
            rates[warps] = blocks * 128 * iters / (ms / 1e3)
        peaks, _ = _peaks()
        mhz = float(peaks.get("sm_max_mhz", 2070.0))
        # XORs and rotates have only the ALU pipe (16 lanes per scheduler): 456 per compression
        alu_bound = sms * mhz * 1e6 * 64 / 456
        line = {"mode": "ceiling", "metric": "compressions/s, messages in registers (keyed BLAKE3 compression, 1 GB300)",
                "value": rates[20] / 1e9, "unit": "G compressions/s",
                "by_warps_per_sm": {str(k): v / 1e9 for k, v in rates.items()},
                "alu_pipe_bound": alu_bound / 1e9, "frac_of_alu_pipe_bound": rates[20] / alu_bound,
                "implied_digest_GBps": rates[20] * 1024 / 17 / 1e9,
                "config": {"kernel": "compress_rate_kernel (blake3_selftest_compress_rate)",
                           "iters_per_thread": iters, "threads_per_cta": 128,
                           "implied": "16 leaf compressions + 1 parent per 1024-byte chunk"}}
    elif args.mode == "latency":
        # several lanes per chunk (the page's future-work item): the latency of a chain of
        # dependent compressions in one warp, one lane per chain against four lanes per
        # chain (the state split by columns, shuffles for the diagonal step)
        key = workloads.key_bytes(11)
        peaks, _ = _peaks()
        mhz = float(peaks.get("sm_max_mhz", 2070.0))
        res = {}
        for lanes in (1, 4):
            cvs = torch.zeros((32 // lanes, 32), dtype=torch.uint8, device="cuda")
            cycles = torch.zeros(1, dtype=torch.int64, device="cuda")
            per = {}
            for chain in (16, 1024):
                for _ in range(args.warmup):
                    binding.blake3_selftest_compress_latency(lanes, chain, key, cvs, cycles)
                torch.cuda.synchronize()
                cyc = []
                for _ in range(args.steps):
                    binding.blake3_selftest_compress_latency(lanes, chain, key, cvs, cycles)
                    torch.cuda.synchronize()
                    cyc.append(int(cycles.item()))
                c = statistics.median(cyc)
                per[str(chain)] = {"cycles": c, "cycles_per_compression": c / chain,
                                   "us_at_max_clock": c / mhz}
            ms16 = _timed(lambda: binding.blake3_selftest_compress_latency(lanes, 16, key, cvs, cycles),
                          args.steps, args.warmup)
            res[f"{lanes}_lane{'s' if lanes > 1 else ''}_per_chunk"] = {
                "chains_per_warp": 32 // lanes, "by_chain": per, "launch_us_chain16_events": ms16 * 1e3}
        one = res["1_lane_per_chunk"]["by_chain"]["1024"]["cycles_per_compression"]
        four = res["4_lanes_per_chunk"]["by_chain"]["1024"]["cycles_per_compression"]
        line = {"mode": "latency", "metric": "cycles per dependent compression, one warp (keyed BLAKE3, 1 GB300)",
                "value": four / one, "unit": "4-lane latency / 1-lane latency", "results": res,
                "config": {"kernel": "compress_latency_kernel (blake3_selftest_compress_latency)",
                           "clock_for_us": f"{mhz:.0f} MHz (maximum SM clock)",
                           "chunk_latency_16_blocks_us": {"1 lane": res["1_lane_per_chunk"]["by_chain"]["16"]
                                                          ["us_at_max_clock"],
                                                          "4 lanes": res["4_lanes_per_chunk"]["by_chain"]["16"]
                                                          ["us_at_max_clock"]}}}
    else:  # small: the 1 MiB digest, per call and replayed from a CUDA graph
        w = workloads.WORKLOADS["1MiB"]
        d = w.data(device="cuda")
        key = w.key()
        out32 = torch.empty(32, dtype=torch.uint8, device="cuda")
        ms_call = _timed(lambda: binding.blake3_keyed_hash(d, key, out=out32), args.steps, args.warmup)
        ws = torch.empty(max(16, binding.blake3_workspace_size(d.numel())), dtype=torch.uint8, device="cuda")
        per_graph = 50
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                binding.blake3_keyed_hash_ws(d, key, ws, out=out32)
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for _ in range(per_graph):
                binding.blake3_keyed_hash_ws(d, key, ws, out=out32)
        ms_graph = _timed(graph.replay, max(3, args.steps // per_graph), 2) / per_graph
        if bytes(out32.cpu().numpy()) != bytes(binding.blake3_keyed_hash(d, key).cpu().numpy()):
            raise RuntimeError("graph-replayed digest differs")
        # the same with the fused final reduction (one launch + a 4-byte memset)
        binding.blake3_set_option(binding.B3G_OPT_FUSED_FINAL, 1)
        try:
            with torch.cuda.stream(s):
                for _ in range(3):
                    binding.blake3_keyed_hash_ws(d, key, ws, out=out32)
            torch.cuda.current_stream().wait_stream(s)
            graph_f = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph_f, stream=s):
                for _ in range(per_graph):
                    binding.blake3_keyed_hash_ws(d, key, ws, out=out32)
            ms_fused = _timed(graph_f.replay, max(3, args.steps // per_graph), 2) / per_graph
        finally:
            binding.blake3_set_option(binding.B3G_OPT_FUSED_FINAL, 0)
        line = {"mode": "small", "metric": "GB/s hashed, 1 MiB input (keyed BLAKE3, 1 GB300)",
                "value": d.numel() / ms_graph / 1e6, "unit": "GB/s", "us_per_digest_graph": ms_graph * 1e3,
                "us_per_call_eager": ms_call * 1e3, "eager_GBps": d.numel() / ms_call / 1e6,
                "us_per_digest_graph_fused_final": ms_fused * 1e3,
                "config": {"workload": "1MiB uniform seed 0, key seed 1",
                           "graph": f"{per_graph} blake3_keyed_hash_ws calls per CUDA graph"}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=7)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration measurements")
    ap.add_argument("--no-oracle-check", action="store_true", help="skip the oracle check of the headline digest")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--mode", choices=["headline", "xof", "stream", "small", "default", "ceiling", "latency"],
                    default="headline")
    ap.add_argument("--xof-bytes", type=int, default=1 << 32)
    ap.add_argument("--segment-bytes", type=int, default=(256 << 20) + 777)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.mode != "headline":
        return run_mode(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

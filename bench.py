#!/usr/bin/env python3
"""Benchmark: U32 exclusive scan, in place, n = 2^28, on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one call of scan_exclusive_u32 on a resident 1 GiB array of
uniform u32 (seed 2), in place, with its total; the same buffer is rescanned
every step (identical traffic; the 1 GiB input is far larger than the
129 MB L2, so no flush is needed between steps). Rank 0 prints one JSON line.

value      elements scanned per second over all ranks (Gelem/s), device-timed
           with CUDA events on the launching stream, max over ranks.
roofline   the scan kernel's algorithmic bytes (4 read + 4 written per
           element) over its measured time, against the measured HBM copy
           peak in MEASURED_PEAKS.json (fallback 6800 GB/s when absent).
e2e        the same metric through the same C-ABI call, with a pinned host
           input copied in and the result and total copied out every step.
cpu_baseline  the CPU oracle (one thread, as it stands) on a bounded sample.

--impl reference times that oracle alone on the host cores (rank 0 only).
Under torchrun each rank scans its own array on its own GPU (independent
replicas: weak scaling, no data-path collective).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import pathlib
import shutil
import subprocess
import sys
import threading
import time

ROOT = pathlib.Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

N = 1 << 28
SEED = 2
BYTES_PER_ELEM = 8  # one 4-byte read and one 4-byte write per element
METRIC = "U32 exclusive scan Gelem/s and HBM GB/s (fraction of peak) at n=2^28, 1 GB300"
UNIT = "Gelem/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = "u32 exclusive scan in place + total, n=2^28, uniform u32 seed 2"
KERNEL_SOURCES = ["u32_prefix_scan_gb300/csrc/scan.cu", "u32_prefix_scan_gb300/csrc/internal.cuh"]
TRAFFIC_FILE = ROOT / "profiles" / "scan_exclusive_u32_n2p28.traffic.json"
REF_SAMPLE = 1 << 24  # elements per reference-arm step


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--log2n", type=int, default=28,
                   help="array size 2^log2n (28 is the benchmark; smaller sizes are for profiler captures)")
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be at least 3")
    if a.steps < 1:
        p.error("--steps must be at least 1")
    return a


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def load_peak():
    f = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(f.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_traffic():
    """ncu DRAM bytes per launch, if captured for the current kernel source."""
    try:
        d = json.loads(TRAFFIC_FILE.read_text())
    except Exception:
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    return float(d["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, kept for the
    timed window only."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if exe is None:
            return self
        self.proc = subprocess.Popen(
            [exe, f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"],
            stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        rows = [l for (t, l) in self.lines if self.t0 is None or (self.t0 - 0.06 <= t <= self.t1 + 0.06)]
        if not rows and self.lines:
            rows = [self.lines[-1][1]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[3:7]):
                if flag.lower() in ("active", "1"):
                    reasons.add(name)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def time_oracle_scan(host_u32, seconds: float):
    """The oracle's exclusive scan (one thread), repeated in place over the
    given array until `seconds` have passed. Returns elements/s and reps."""
    import ctypes

    import oracle

    lib = oracle._load()
    ptr = host_u32.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32))
    n = host_u32.size
    reps, t0 = 0, time.perf_counter()
    while True:
        lib.oracle_scan_exclusive_u32(ptr, n)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return n * reps / el, reps, el


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on the host cores, rank 0 only."""
    if rank != 0:
        return None
    import numpy as np

    from u32_prefix_scan_gb300 import inputs

    import oracle

    oracle.build()
    sample = min(N, REF_SAMPLE)
    host = inputs.scan_values(sample, SEED)
    import ctypes

    lib = oracle._load()
    ptr = host.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32))
    for _ in range(args.warmup):
        lib.oracle_scan_exclusive_u32(ptr, sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        lib.oracle_scan_exclusive_u32(ptr, sample)
    el = time.perf_counter() - t0
    value = sample * args.steps / el / 1e9
    desc = f"oracle_scan_exclusive_u32 on the first 2^{sample.bit_length() - 1} elements of the workload per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "n": N, "seed": SEED, "sample_per_step": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ours(args, rank, local_rank, world):
    import numpy as np
    import torch

    import u32_prefix_scan_gb300 as u
    from u32_prefix_scan_gb300 import _native, inputs
    from u32_prefix_scan_gb300 import build as native_build

    native_build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()

    host = inputs.scan_values(N, SEED)
    data = torch.from_numpy(host.view(np.int32)).to(dev)
    total = torch.empty(1, dtype=torch.int32, device=dev)
    ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_SCAN, N), dev)

    for _ in range(args.warmup):
        u.scan_exclusive_u32(data, total, workspace=ws)
    u.check(workspace=ws)

    sampler = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.15)
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        u.scan_exclusive_u32(data, total, workspace=ws)
    end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    sampler.window(w0, w1)
    clocks = sampler.stop()
    u.check(workspace=ws)
    ms = start.elapsed_time(end) / args.steps
    ms_max = max_over_ranks(ms, world)

    # end to end through the C ABI: pinned host in -> scan -> host out
    h_in = torch.from_numpy(host.view(np.int32)).pin_memory()
    h_out = torch.empty(N, dtype=torch.int32).pin_memory()
    h_tot = torch.empty(1, dtype=torch.int32).pin_memory()
    for _ in range(2):
        data.copy_(h_in, non_blocking=True)
        u.scan_exclusive_u32(data, total, workspace=ws)
        h_out.copy_(data, non_blocking=True)
        h_tot.copy_(total, non_blocking=True)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(args.e2e_steps):
        data.copy_(h_in, non_blocking=True)
        u.scan_exclusive_u32(data, total, workspace=ws)
        h_out.copy_(data, non_blocking=True)
        h_tot.copy_(total, non_blocking=True)
    e_end.record(stream)
    torch.cuda.synchronize()
    u.check(workspace=ws)
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / args.e2e_steps, world)

    # sanity property of the copied-back result (exclusive scan of host):
    # out[0] = 0 and out[j+1] - out[j] = in[j] (mod 2^32) on a prefix
    k = 1 << 20
    got = h_out[:k].numpy().view(np.uint32)
    if got[0] != 0 or not np.array_equal(got[1:] - got[:-1], host[: k - 1]):
        raise SystemExit("bench: e2e result is not the exclusive scan of its input")

    peak, peak_kind = load_peak()
    achieved = BYTES_PER_ELEM * N / (ms * 1e-3) / 1e9
    traffic = load_traffic()
    result = {
        "metric": METRIC,
        "value": world * N / (ms_max * 1e-3) / 1e9,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if N == 1 << 28 else f"profiling case n=2^{args.log2n}", "n": N,
                   "seed": SEED, "per_rank": "one independent array per GPU",
                   "l2": "input 1 GiB > 129 MB L2; no flush between steps"},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic, "algorithmic_bytes_per_launch": BYTES_PER_ELEM * N,
                     "kernel": "scan_u32_persistent<512,8,2,1,exclusive>"},
        "e2e": {"value": world * N / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": 4 * N, "d2h_bytes_per_step": 4 * N + 4},
        "clocks": clocks,
        "gpu_launches": args.steps,
    }
    if rank == 0 and not args.no_cpu_baseline:
        sample = host.copy()
        v, reps, el = time_oracle_scan(sample, args.cpu_seconds)
        result["cpu_baseline"] = {"value": v / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
                                  "sample": f"oracle_scan_exclusive_u32 over the full 2^28 workload, "
                                            f"in place, {reps} repetitions in {el:.1f} s"}
    return result


def main(argv=None):
    global N
    args = parse_args(argv)
    N = 1 << args.log2n
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        # rank 0 alone times the oracle; other ranks exit without work
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend="nccl")
    out = run_ours(args, rank, local_rank, world)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

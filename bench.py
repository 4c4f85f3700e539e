#!/usr/bin/env python3
"""Benchmark of the U32 scan primitives on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--op OP] [--heads geometric|regular4]

Default (--op scan_exclusive): one step is one call of scan_exclusive_u32 on
a resident 1 GiB array (n = 2^28 uniform u32, seed 2), in place, with its
total; the same buffer is rescanned every step (identical traffic; the input
is far larger than the 129 MB L2, so no flush is needed between steps).
Other ops time the other primitives on their own workloads:

  scan_inclusive  scan_inclusive_u32, n = 2^28, seed 2
  scan_op         scan_u32_op under --monoid (add mul and or xor min max),
                  exclusive or --inclusive, n = 2^28, seed 2
  segscan         segscan_inclusive_u32 in place, n = 2^26, values seed 3,
                  heads --heads (Bernoulli 2^-10 or every 4th index)
  segscan_sums    the same, also writing every segment's sum and the count
  segreduce       segreduce_u32: sums and count only
  compact         compact_indices_u32, n = 2^27 int32 flags, keep
                  probability --p (0.1 or 0.9), seed 4; --project values
                  or nonzero times compact_values_u32 (values u32(4,0,i))
  radix           radix_sort_perm_u32, n = 2^25 keys seed 5, uniform u32
                  or (--ties) in [0, 256); --sort pairs|keys times
                  radix_sort_u32 writing sorted keys (+ perm unless keys)
  scan64          scan_u64_op in place, n = 2^27 uint64, --monoid64 (add),
                  exclusive or --inclusive
  runs            runs_layout_u32 + runs_owner_u32, n = 2^25 owners, counts
                  u32(6,0,i) >> 29 in [0, 8) or (--skewed) one owner in 16
                  holding up to 63 entries

Rank 0 prints one JSON line.

value      elements processed per second over all ranks (Gelem/s), timed
           with CUDA events on the launching stream, max over ranks.
roofline   algorithmic bytes of one launch over its measured time, against
           the measured HBM copy peak in MEASURED_PEAKS.json (fallback
           6800 GB/s when absent); also against a device copy timed in the
           same run (copy_gbs_same_run) and the nominal 7900 GB/s. For a
           step of several calls the dominant kernel is bracketed by its
           own events (kernel_ms).
e2e        the same metric end to end from pinned host memory: the add
           scans call scan_{exclusive,inclusive}_u32_host, which streams the
           host array through the device in chunks (copies in, scans and
           copies out overlapped); the other ops copy their inputs in, make
           the same C-ABI call and copy their outputs out, every step.
cpu_baseline  the CPU oracle (one thread, as it stands) on a bounded sample.
library_context  (--library-context) PyTorch's CUDA cumsum over the
           same values (the add scans), or its stable sort of the same keys
           (radix), timed the same way, with a bit-for-bit comparison
           against this library's result: context, not a baseline.

--impl reference times that oracle alone on the host cores (rank 0 only).
Under torchrun each rank runs its own replica of the workload on its own GPU
(independent replicas: weak scaling, no data-path collective).
"""

from __future__ import annotations

import argparse
import ctypes
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

UNIT = "Gelem/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000  # GB300's L2
REF_SAMPLE = 1 << 24  # elements per reference-arm step


# ------------------------------------------------------------------ ops ----

class Op:
    """One benchmarked primitive on its workload."""

    name = ""
    metric = ""
    kernel = ""
    kernel_sources: list = []
    log2n = 28
    launches_per_step = 1  # this library's kernels launched by one step

    def __init__(self, args):
        self.args = args
        self.n = 1 << (args.log2n if args.log2n is not None else self.log2n)

    @property
    def traffic_file(self):
        return ROOT / "profiles" / f"{self.name}_n2p{self.log2n}.traffic.json"

    def workload(self) -> str:
        raise NotImplementedError

    def algorithmic_bytes(self) -> int:
        raise NotImplementedError

    def is_marked(self) -> bool:
        """Whether a step brackets its dominant kernel with events (step_marked)."""
        return hasattr(self, "step_marked")


class ScanOp(Op):
    log2n = 28
    kernel_sources = ["u32_prefix_scan_gb300/csrc/scan.cu", "u32_prefix_scan_gb300/csrc/internal.cuh"]

    def __init__(self, args, inclusive: bool, monoid: str = "add"):
        super().__init__(args)
        self.inclusive = inclusive
        self.monoid = monoid
        # under torchrun: rank r scans its shard of one array of N * n elements
        self.world, self.rank = getattr(args, "world", 1), getattr(args, "rank", 0)
        self.sharded = self.world > 1 and monoid == "add"
        if self.sharded:
            self.launches_per_step = 3  # fold, scan of the gathered sums, scan from the carry-in
        form = "inclusive" if inclusive else "exclusive"
        self.name = f"scan_{form}_u32" if monoid == "add" else f"scan_{monoid}_{form}_u32"
        what = "" if monoid == "add" else f"{monoid} "
        self.metric = f"U32 {what}{form} scan Gelem/s and HBM GB/s (fraction of peak) at n=2^28, 1 GB300"
        self.kernel = f"scan_u32_persistent<512,8,2,1,{form},{monoid}> (bulk-copy stores)"

    def workload(self):
        form = "inclusive" if self.inclusive else "exclusive"
        what = "" if self.monoid == "add" else f"{self.monoid}-"
        lg = self.n.bit_length() - 1
        if self.sharded:
            return (f"u32 {form} scan in place + total of one array of {self.world} x 2^{lg} elements (uniform u32 "
                    f"seed 2), sharded: rank r holds elements [r 2^{lg}, (r+1) 2^{lg})")
        return f"u32 {what}{form} scan in place + total, n=2^{lg}, uniform u32 seed 2"

    def algorithmic_bytes(self):
        return 8 * self.n  # read 4 + write 4 per element (the scan kernel; the sharded fold reads 4 more)

    def host_inputs(self):
        from u32_prefix_scan_gb300 import inputs

        if self.sharded:
            return {"data": inputs.splitmix_u32(2, 0, self.n, start=self.rank * self.n)}
        return {"data": inputs.scan_values(self.n, 2)}

    def is_marked(self) -> bool:
        return self.sharded

    def setup(self, dev, host):
        import numpy as np
        import torch

        import u32_prefix_scan_gb300 as u
        from u32_prefix_scan_gb300 import _native

        self.u = u
        if self.monoid == "add":
            self.fn = u.scan_inclusive_u32 if self.inclusive else u.scan_exclusive_u32
        else:
            self.fn = lambda d, t, workspace: u.scan_u32_op(d, self.monoid, self.inclusive, t, workspace=workspace)
        self.data = torch.from_numpy(host["data"].view(np.int32)).to(dev)
        self.total = torch.empty(1, dtype=torch.int32, device=dev)
        lib = _native.lib()
        self.ws = u.Workspace(max(lib.u32scan_workspace_bytes(_native.OP_SCAN, self.n),
                                  lib.u32scan_workspace_bytes(_native.OP_REDUCE, self.n)), dev)
        if self.sharded:
            from u32_prefix_scan_gb300 import shard

            self.shard = shard
            self.steps = shard.KernelSteps(workspace=self.ws)
        self.pinned_in = {"data": torch.from_numpy(host["data"].view(np.int32)).pin_memory()}
        self.pinned_out = {"data": torch.empty(self.n, dtype=torch.int32).pin_memory(),
                           "total": torch.empty(1, dtype=torch.int32).pin_memory()}
        if self.monoid == "add":
            self.host_fn = u.scan_inclusive_u32_host if self.inclusive else u.scan_exclusive_u32_host
            self.ws_host = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_SCAN_HOST, self.n), dev)

    def step(self):
        if self.sharded:
            self.total = self.shard.sharded_scan(self.data, self.inclusive, steps=self.steps)
        else:
            self.fn(self.data, self.total, workspace=self.ws)

    def step_marked(self, before, after):
        """The sharded step with events around its scan from the carry-in,
        the kernel that moves 8 of its 12 bytes an element."""
        self.total = self.shard.sharded_scan(self.data, self.inclusive, steps=self.steps, marks=(before, after))

    def e2e_step(self):
        if self.sharded:  # the shard in from pinned host memory, the sharded scan, the shard and total out
            self.data.copy_(self.pinned_in["data"], non_blocking=True)
            self.step()
            self.pinned_out["data"].copy_(self.data, non_blocking=True)
            self.pinned_out["total"].copy_(self.total, non_blocking=True)
            return 4 * self.n, 4 * self.n + 4
        if self.monoid == "add":  # host array in, host array out, through the device in overlapped chunks
            self.host_fn(self.pinned_in["data"], self.pinned_out["data"], self.pinned_out["total"],
                         workspace=self.ws_host)
            return 4 * self.n, 4 * self.n + 4
        self.data.copy_(self.pinned_in["data"], non_blocking=True)
        self.step()
        self.pinned_out["data"].copy_(self.data, non_blocking=True)
        self.pinned_out["total"].copy_(self.total, non_blocking=True)
        return 4 * self.n, 4 * self.n + 4

    def check_e2e(self, host):
        # consecutive differences of the copied-back scan give the input
        import numpy as np

        if self.monoid != "add":
            return True  # checked bit for bit by the GPU tests; no cheap property here
        k = min(self.n, 1 << 20)
        got = self.pinned_out["data"][:k].numpy().view(np.uint32)
        a = host["data"][:k]
        if self.sharded:  # the shard starts from its carry-in; the total is the whole array's
            return np.array_equal(got[1:] - got[:-1], a[1:] if self.inclusive else a[:-1])
        total = int(self.pinned_out["total"].numpy().view(np.uint32)[0])
        if total != int(host["data"].sum(dtype=np.uint64)) % (1 << 32):
            return False
        if self.inclusive:
            return got[0] == a[0] and np.array_equal(got[1:] - got[:-1], a[1:])
        return got[0] == 0 and np.array_equal(got[1:] - got[:-1], a[:-1])

    def library_context(self, host, steps: int):
        """PyTorch's own CUDA scan of the same values, timed the same way, for
        context: torch.cumsum over int32 with an int32 result wraps exactly
        as the U32 inclusive scan does (two's-complement addition), out of
        place, so it moves the same 8 B/element. Its bits are compared with
        this library's inclusive scan of the same input."""
        import numpy as np
        import torch

        x = torch.from_numpy(host["data"].view(np.int32)).to(self.data.device)
        y = torch.empty_like(x)
        z = x.clone()
        self.u.scan_inclusive_u32(z, workspace=self.ws)
        torch.cumsum(x, 0, dtype=torch.int32, out=y)
        torch.cuda.synchronize()
        same = bool(torch.equal(y, z))
        del z
        for _ in range(3):
            torch.cumsum(x, 0, dtype=torch.int32, out=y)
        stream = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(steps):
            torch.cumsum(x, 0, dtype=torch.int32, out=y)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        return {"call": "torch.cumsum(int32 values, dtype=int32, out=...) on the same device array", "ms_per_step": ms,
                "value": self.n / (ms * 1e-3) / 1e9, "unit": UNIT, "hbm_gbs": 8 * self.n / (ms * 1e-3) / 1e9,
                "bits_equal_to_scan_inclusive_u32": same}

    def oracle_step(self, lib, arrays):
        ptr = arrays["data"].ctypes.data_as(ctypes.POINTER(ctypes.c_uint32))
        if self.monoid != "add":
            codes = {"add": 0, "mul": 1, "and": 2, "or": 3, "xor": 4, "min": 5, "max": 6}
            lib.oracle_scan_op_u32(codes[self.monoid], int(self.inclusive), ptr, arrays["data"].size)
            return
        f = lib.oracle_scan_inclusive_u32 if self.inclusive else lib.oracle_scan_exclusive_u32
        f(ptr, arrays["data"].size)


class Scan64Op(Op):
    """scan_u64_op in place on a 2^27-element (1 GiB) uint64 row."""

    log2n = 27
    kernel_sources = ["u32_prefix_scan_gb300/csrc/scan64.cu", "u32_prefix_scan_gb300/csrc/internal.cuh"]

    def __init__(self, args):
        super().__init__(args)
        self.inclusive = args.inclusive
        self.monoid = args.monoid64
        form = "inclusive" if self.inclusive else "exclusive"
        self.name = f"scan_u64_{self.monoid}_{form}"
        self.metric = f"U64 {self.monoid} {form} scan Gelem/s and HBM GB/s (fraction of peak) at n=2^27, 1 GB300"
        self.kernel = f"scan_u64_persistent<512,8,2,{form},{self.monoid}> (bulk-copy stores)"

    def workload(self):
        form = "inclusive" if self.inclusive else "exclusive"
        return (f"u64 {self.monoid}-{form} scan in place + fold, n=2^{self.n.bit_length() - 1}, "
                f"uniform u64 seed 2 (two u32 draws per element)")

    def algorithmic_bytes(self):
        return 16 * self.n  # read 8 + write 8 per element

    def host_inputs(self):
        from u32_prefix_scan_gb300 import inputs

        return {"data": inputs.scan_values_u64(self.n, 2)}

    def setup(self, dev, host):
        import numpy as np
        import torch

        import u32_prefix_scan_gb300 as u
        from u32_prefix_scan_gb300 import _native

        self.u = u
        self.data = torch.from_numpy(host["data"].view(np.int64)).to(dev)
        self.total = torch.empty(1, dtype=torch.int64, device=dev)
        self.ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_SCAN64, self.n), dev)
        self.pinned_in = {"data": torch.from_numpy(host["data"].view(np.int64)).pin_memory()}
        self.pinned_out = {"data": torch.empty(self.n, dtype=torch.int64).pin_memory(),
                           "total": torch.empty(1, dtype=torch.int64).pin_memory()}

    def step(self):
        self.u.scan_u64_op(self.data, self.monoid, self.inclusive, self.total, workspace=self.ws)

    def e2e_step(self):
        self.data.copy_(self.pinned_in["data"], non_blocking=True)
        self.step()
        self.pinned_out["data"].copy_(self.data, non_blocking=True)
        self.pinned_out["total"].copy_(self.total, non_blocking=True)
        return 8 * self.n, 8 * self.n + 8

    def check_e2e(self, host):
        import numpy as np

        if self.monoid != "add":
            return True  # checked bit for bit by the GPU tests
        k = min(self.n, 1 << 20)
        got = self.pinned_out["data"][:k].numpy().view(np.uint64)
        a = host["data"][:k]
        if self.inclusive:
            return got[0] == a[0] and np.array_equal(got[1:] - got[:-1], a[1:])
        return got[0] == 0 and np.array_equal(got[1:] - got[:-1], a[:-1])

    def oracle_step(self, lib, arrays):
        codes = {"add": 0, "mul": 1, "and": 2, "or": 3, "xor": 4, "min": 5, "max": 6}
        a = arrays["data"]
        lib.oracle_scan_op_u64(codes[self.monoid], int(self.inclusive),
                               a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), a.size)


class SegOp(Op):
    log2n = 26
    kernel_sources = ["u32_prefix_scan_gb300/csrc/segscan.cu", "u32_prefix_scan_gb300/csrc/internal.cuh"]

    def __init__(self, args, mode: str):
        super().__init__(args)
        self.mode = mode  # segscan | segscan_sums | segreduce
        self.heads = args.heads
        self.fbytes = 1 if args.u8heads else 4  # bytes per head flag
        self.name = f"{mode}_{self.heads}" + ("_u8heads" if args.u8heads else "")
        what = {"segscan": "segmented inclusive scan", "segscan_sums": "segmented inclusive scan + segment sums",
                "segreduce": "per-segment reduce"}[mode]
        lengths = "geometric lengths mean 1024" if self.heads == "geometric" else "2^24 segments of length 4"
        fl = ", u8 head flags" if args.u8heads else ""
        self.metric = f"U32 {what} Gelem/s and HBM GB/s (fraction of peak) at n=2^26 ({lengths}{fl}), 1 GB300"
        kind = {"segscan": "true,false", "segscan_sums": "true,true", "segreduce": "false,true"}[mode]
        # (u32x4 a lane, ring stages, output buffer) as the library picks them
        if mode == "segreduce":
            r, stages, buf = 7, 3 if args.u8heads else 2, 0
        else:
            r, stages, buf = 7 if args.u8heads else 5, 2, 1
        ftype = "uint8" if args.u8heads else "int32"
        self.kernel = f"segscan_lanes_persistent<512,{r},{stages},{kind},{ftype},{buf}>"
        self.nseg = None
        # under torchrun, the segmented scan with int32 flags: rank r scans its
        # shard of one array of N * n elements
        self.world, self.rank = getattr(args, "world", 1), getattr(args, "rank", 0)
        self.sharded = self.world > 1 and mode == "segscan" and not args.u8heads
        if self.sharded:
            self.launches_per_step = 6  # scan, summary, carries, first head, fix (+ its init)

    def workload(self):
        lengths = "Bernoulli(2^-10) heads" if self.heads == "geometric" else "a head every 4th index"
        ftype = "u8" if self.fbytes == 1 else "int32"
        lg = self.n.bit_length() - 1
        if self.sharded:
            return (f"u32 segmented scan of one array of {self.world} x 2^{lg} elements, values uniform u32 seed 3, "
                    f"int32 head flags: {lengths}; sharded: rank r holds elements [r 2^{lg}, (r+1) 2^{lg})")
        return (f"u32 {self.mode} n=2^{lg}, values uniform u32 seed 3, {ftype} head "
                f"flags: {lengths}")

    def is_marked(self) -> bool:
        return self.sharded

    def algorithmic_bytes(self):
        n, nseg, fb = self.n, self.nseg, self.fbytes
        if self.mode == "segscan":
            return (8 + fb) * n  # values 4 + flags read, values 4 written
        if self.mode == "segscan_sums":
            return (8 + fb) * n + 4 * nseg + 4
        return (4 + fb) * n + 4 * nseg + 4  # segreduce: values + flags read, one sum per segment

    def host_inputs(self):
        import numpy as np

        from u32_prefix_scan_gb300 import inputs

        start = self.rank * self.n if self.sharded else 0
        f = (inputs.segment_heads_geometric(self.n, 3, start=start) if self.heads == "geometric"
             else inputs.segment_heads_regular(self.n, 4))  # n is a multiple of 4: every shard alike
        self.nseg = int(np.count_nonzero(f))
        if self.fbytes == 1:
            f = f.astype(np.uint8)
        return {"data": inputs.splitmix_u32(3, 0, self.n, start=start), "flags": f}

    def setup(self, dev, host):
        import numpy as np
        import torch

        import u32_prefix_scan_gb300 as u
        from u32_prefix_scan_gb300 import _native

        self.u = u
        self.data = torch.from_numpy(host["data"].view(np.int32)).to(dev)
        self.flags = torch.from_numpy(host["flags"]).to(dev)
        self.sums = torch.empty(self.nseg, dtype=torch.int32, device=dev) if self.mode != "segscan" else None
        self.count = torch.empty(1, dtype=torch.int32, device=dev)
        self.ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_SEGSCAN, self.n), dev)
        if self.sharded:
            from u32_prefix_scan_gb300 import shard

            self.shard = shard
            self.steps = shard.KernelSteps(workspace=self.ws)
        self.pinned_in = {"data": torch.from_numpy(host["data"].view(np.int32)).pin_memory(),
                          "flags": torch.from_numpy(host["flags"]).pin_memory()}
        self.pinned_out = {"count": torch.empty(1, dtype=torch.int32).pin_memory()}
        if self.mode != "segreduce":
            self.pinned_out["data"] = torch.empty(self.n, dtype=torch.int32).pin_memory()
        if self.sums is not None:
            self.pinned_out["sums"] = torch.empty(self.nseg, dtype=torch.int32).pin_memory()

    def step(self):
        if self.sharded:
            self.count = self.shard.sharded_segscan(self.data, self.flags, steps=self.steps)
        elif self.mode == "segreduce":
            self.u.segreduce_u32(self.data, self.flags, self.sums, self.count, workspace=self.ws)
        else:
            self.u.segscan_inclusive_u32(self.data, self.flags, self.sums, self.count, workspace=self.ws)

    def step_marked(self, before, after):
        """The sharded step with events around the shard's own segmented scan,
        the kernel that moves its 12 bytes an element."""
        self.count = self.shard.sharded_segscan(self.data, self.flags, steps=self.steps, marks=(before, after))

    def e2e_step(self):
        self.data.copy_(self.pinned_in["data"], non_blocking=True)
        self.flags.copy_(self.pinned_in["flags"], non_blocking=True)
        self.step()
        d2h = 4
        self.pinned_out["count"].copy_(self.count, non_blocking=True)
        if "data" in self.pinned_out:
            self.pinned_out["data"].copy_(self.data, non_blocking=True)
            d2h += 4 * self.n
        if "sums" in self.pinned_out:
            self.pinned_out["sums"].copy_(self.sums, non_blocking=True)
            d2h += 4 * self.nseg
        return (4 + self.fbytes) * self.n, d2h

    def check_e2e(self, host):
        if self.sharded:  # the whole array's count: at least this shard's heads
            return int(self.pinned_out["count"][0]) >= self.nseg
        return int(self.pinned_out["count"][0]) == self.nseg

    def oracle_step(self, lib, arrays):
        u32p, i32p = ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_int32)
        if arrays["flags"].itemsize != 4:
            import numpy as np

            arrays["flags"] = arrays["flags"].astype(np.int32)  # the oracle reads int32 flags
        a, f = arrays["data"], arrays["flags"]
        if self.mode == "segscan":
            lib.oracle_segscan_inclusive_u32(a.ctypes.data_as(u32p), f.ctypes.data_as(i32p), a.size)
            return
        if "sums" not in arrays:
            import numpy as np

            arrays["sums"] = np.zeros(max(a.size, 1), dtype=np.uint32)
        lib.oracle_segreduce_u32(a.ctypes.data_as(u32p), f.ctypes.data_as(i32p), a.size,
                                 arrays["sums"].ctypes.data_as(u32p))
        if self.mode == "segscan_sums":
            lib.oracle_segscan_inclusive_u32(a.ctypes.data_as(u32p), f.ctypes.data_as(i32p), a.size)


class CompactOp(Op):
    log2n = 27
    kernel_sources = ["u32_prefix_scan_gb300/csrc/compact.cu", "u32_prefix_scan_gb300/csrc/internal.cuh"]

    def __init__(self, args):
        super().__init__(args)
        self.p = args.p
        self.name = f"compact_p{self.p}"
        self.metric = (f"stream compaction Gelem/s and HBM GB/s (fraction of peak) at n=2^27, "
                       f"Bernoulli p={self.p} int32 flags, 1 GB300")
        self.kernel = "compact_persistent<512,8,2>"
        # under torchrun: rank r compacts its shard of one array of N * n flags
        self.world, self.rank = getattr(args, "world", 1), getattr(args, "rank", 0)
        self.sharded = self.world > 1
        if self.sharded:
            self.launches_per_step = 4  # count, two scans of the gathered words, compaction from the carry-ins

    def workload(self):
        lg = self.n.bit_length() - 1
        if self.sharded:
            return (f"compaction of one array of {self.world} x 2^{lg} int32 flags, Bernoulli p={self.p} (seed 4), "
                    f"sharded: rank r holds flags [r 2^{lg}, (r+1) 2^{lg}); whole-array offsets and indices, counts")
        return (f"compaction of n=2^{lg} int32 flags, Bernoulli p={self.p} (seed 4): "
                f"inclusive offsets, kept indices with -1 tail, count")

    def is_marked(self) -> bool:
        return self.sharded

    def algorithmic_bytes(self):
        return 12 * self.n + 4  # flags read; offsets and one index slot written per element; the count

    def host_inputs(self):
        from u32_prefix_scan_gb300 import inputs

        return {"flags": inputs.compact_flags(self.n, 4, self.p, start=self.rank * self.n)}

    def setup(self, dev, host):
        import torch

        import u32_prefix_scan_gb300 as u
        from u32_prefix_scan_gb300 import _native

        self.u = u
        if self.sharded:
            from u32_prefix_scan_gb300 import shard

            self.shard = shard
        self.flags = torch.from_numpy(host["flags"]).to(dev)
        self.offsets = torch.empty(self.n, dtype=torch.int32, device=dev)
        self.indices = torch.empty(self.n, dtype=torch.int32, device=dev)
        self.count = torch.empty(1, dtype=torch.int32, device=dev)
        lib = _native.lib()
        self.ws = u.Workspace(max(lib.u32scan_workspace_bytes(_native.OP_COMPACT, self.n),
                                  lib.u32scan_workspace_bytes(_native.OP_SCAN, self.world),
                                  lib.u32scan_workspace_bytes(_native.OP_REDUCE, self.n)), dev)
        if self.sharded:
            self.steps = shard.KernelSteps(workspace=self.ws)
        self.pinned_in = {"flags": torch.from_numpy(host["flags"]).pin_memory()}
        self.pinned_out = {k: torch.empty(self.n, dtype=torch.int32).pin_memory() for k in ("offsets", "indices")}
        self.pinned_out["count"] = torch.empty(1, dtype=torch.int32).pin_memory()

    def step(self):
        if self.sharded:
            self.offsets, self.indices, self.count, _ = self.shard.sharded_compact(self.flags, steps=self.steps)
        else:
            self.u.compact_indices_u32(self.flags, self.offsets, self.indices, self.count, workspace=self.ws)

    def step_marked(self, before, after):
        """The sharded step with events around its compaction from the
        carry-ins, the kernel that moves 12 of its 16 bytes an element."""
        self.offsets, self.indices, self.count, _ = self.shard.sharded_compact(self.flags, steps=self.steps,
                                                                              marks=(before, after))

    def e2e_step(self):
        self.flags.copy_(self.pinned_in["flags"], non_blocking=True)
        self.step()
        self.pinned_out["offsets"].copy_(self.offsets, non_blocking=True)
        self.pinned_out["indices"].copy_(self.indices, non_blocking=True)
        self.pinned_out["count"].copy_(self.count, non_blocking=True)
        return 4 * self.n, 8 * self.n + 4

    def check_e2e(self, host):
        import numpy as np

        c = int(self.pinned_out["count"][0])
        if self.sharded:  # whole-array offsets: the last one exceeds the shard's count by what lies before
            return (c == int(np.count_nonzero(host["flags"])) and int(self.pinned_out["offsets"][-1]) >= c
                    and (c == self.n or int(self.pinned_out["indices"][c]) == -1))
        return (c == int(np.count_nonzero(host["flags"])) and int(self.pinned_out["offsets"][-1]) == c
                and (c == self.n or int(self.pinned_out["indices"][c]) == -1))

    def oracle_step(self, lib, arrays):
        import numpy as np

        i32p = ctypes.POINTER(ctypes.c_int32)
        f = arrays["flags"]
        for k in ("offsets", "indices"):
            if k not in arrays:
                arrays[k] = np.empty(f.size, dtype=np.int32)
        if "count" not in arrays:
            arrays["count"] = np.zeros(1, dtype=np.int32)
        lib.oracle_compact_indices(f.ctypes.data_as(i32p), f.size, arrays["offsets"].ctypes.data_as(i32p),
                                   arrays["indices"].ctypes.data_as(i32p), arrays["count"].ctypes.data_as(i32p))


class CompactValuesOp(Op):
    """compact_values_u32: kept values at the front of out, with int32 flags
    (Bernoulli p) or, with --project nonzero, the values' own non-zero test."""

    log2n = 27
    kernel_sources = ["u32_prefix_scan_gb300/csrc/compact_values.cu", "u32_prefix_scan_gb300/csrc/internal.cuh"]

    def __init__(self, args):
        super().__init__(args)
        self.p = args.p
        self.nonzero = args.project == "nonzero"
        self.name = f"compact_values_{'nonzero' if self.nonzero else 'flags'}_p{self.p}"
        test = "non-zero values" if self.nonzero else "int32 flags"
        self.metric = (f"compaction of values Gelem/s and HBM GB/s (fraction of peak) at n=2^27, "
                       f"kept with probability {self.p} ({test}), 1 GB300")
        self.kernel = f"compact_values_persistent<512,8,2,{'false' if self.nonzero else 'true'}>"
        self.kept = None

    def workload(self):
        if self.nonzero:
            src = f"values u32(4,0,i) | 1 where u32(4,1,i) < T_p, else 0 (p={self.p})"
        else:
            src = f"values u32(4,0,i), int32 flags Bernoulli p={self.p} (seed 4)"
        return f"compaction of values, n=2^{self.n.bit_length() - 1}: {src} -> kept values at the front + count"

    def algorithmic_bytes(self):
        # values (and flags) read once; each kept value written once; the count
        return (4 if self.nonzero else 8) * self.n + 4 * self.kept + 4

    def host_inputs(self):
        import numpy as np

        from u32_prefix_scan_gb300 import inputs

        f = inputs.compact_flags(self.n, 4, self.p)
        v = inputs.scan_values(self.n, 4)
        self.kept = int(np.count_nonzero(f))
        if self.nonzero:
            return {"values": np.where(f != 0, v | np.uint32(1), 0).astype(np.uint32)}
        return {"values": v, "flags": f}

    def setup(self, dev, host):
        import numpy as np
        import torch

        import u32_prefix_scan_gb300 as u
        from u32_prefix_scan_gb300 import _native

        self.u = u
        self.values = torch.from_numpy(host["values"].view(np.int32)).to(dev)
        self.flags = None if self.nonzero else torch.from_numpy(host["flags"]).to(dev)
        self.out = torch.empty(self.n, dtype=torch.int32, device=dev)
        self.count = torch.empty(1, dtype=torch.int32, device=dev)
        self.ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_COMPACT, self.n), dev)
        self.pinned_in = {"values": torch.from_numpy(host["values"].view(np.int32)).pin_memory()}
        if self.flags is not None:
            self.pinned_in["flags"] = torch.from_numpy(host["flags"]).pin_memory()
        self.pinned_out = {"out": torch.empty(self.kept, dtype=torch.int32).pin_memory(),
                           "count": torch.empty(1, dtype=torch.int32).pin_memory()}

    def step(self):
        self.u.compact_values_u32(self.values, self.flags, self.out, self.count, workspace=self.ws)

    def e2e_step(self):
        self.values.copy_(self.pinned_in["values"], non_blocking=True)
        if self.flags is not None:
            self.flags.copy_(self.pinned_in["flags"], non_blocking=True)
        self.step()
        self.pinned_out["out"].copy_(self.out[: self.kept], non_blocking=True)
        self.pinned_out["count"].copy_(self.count, non_blocking=True)
        return 4 * self.n * len(self.pinned_in), 4 * self.kept + 4

    def check_e2e(self, host):
        import numpy as np

        v = host["values"]
        keep = v != 0 if self.nonzero else host["flags"] != 0
        k = min(self.kept, 1 << 20)
        return (int(self.pinned_out["count"][0]) == self.kept
                and np.array_equal(self.pinned_out["out"][:k].numpy().view(np.uint32), v[keep][:k]))

    def oracle_step(self, lib, arrays):
        import numpy as np

        u32p, i32p = ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_int32)
        v = arrays["values"]
        if "out" not in arrays:
            arrays["out"] = np.zeros(v.size, dtype=np.uint32)
        f = arrays.get("flags")
        lib.oracle_compact_values_u32(v.ctypes.data_as(u32p), None if f is None else f.ctypes.data_as(i32p), v.size,
                                      arrays["out"].ctypes.data_as(u32p))


class RadixOp(Op):
    log2n = 25
    launches_per_step = 5  # histogram (its last block plans the passes), 4 digit passes (inactive ones return at once)
    kernel_sources = ["u32_prefix_scan_gb300/csrc/radix.cu", "u32_prefix_scan_gb300/csrc/scan.cu",
                      "u32_prefix_scan_gb300/csrc/internal.cuh"]

    OUTPUTS = {"perm": "int32 perm", "pairs": "sorted keys + int32 perm", "keys": "sorted keys"}

    def __init__(self, args):
        super().__init__(args)
        self.ties = args.ties
        self.mode = args.sort
        entry = "radix_sort_perm_u32" if self.mode == "perm" else "radix_sort_u32"
        self.name = entry + ("" if self.mode == "perm" else "_" + self.mode) + ("_ties" if self.ties else "")
        keys = "keys in [0,256)" if self.ties else "uniform u32 keys"
        what = {"perm": "radix-sort permutation", "pairs": "radix sort (keys + permutation)",
                "keys": "radix sort (keys only)"}[self.mode]
        self.metric = f"stable LSD {what} Gelem/s at n=2^25 ({keys}), 1 GB300"
        self.kernel = "radix path: histogram + radix_onesweep_kernel per active 8-bit digit"

    def workload(self):
        keys = "u32(5,0,i) >> 24, in [0,256)" if self.ties else "u32(5,0,i), uniform"
        return f"stable radix sort of n=2^{self.n.bit_length() - 1} u32 keys {keys} -> {self.OUTPUTS[self.mode]}"

    def passes(self):
        return 1 if self.ties else 4  # digits not constant over the keys

    def algorithmic_bytes(self):
        # this design's bytes: a 4-byte histogram read, then per active digit
        # one pass that reads the keys (4) and, when indices are produced,
        # reads them (4, not on the first pass) and writes them (4); keys are
        # written (4) on every pass but the last of the permutation-only sort
        m, n = self.passes(), self.n
        idx = self.mode != "keys"
        total = 4
        for j in range(m):
            total += 4
            if idx:
                total += (4 if j else 0) + 4
            if j < m - 1 or self.mode != "perm":
                total += 4
        return n * total

    def host_inputs(self):
        from u32_prefix_scan_gb300 import inputs

        return {"keys": inputs.radix_keys(self.n, 5, ties=self.ties)}

    def setup(self, dev, host):
        import numpy as np
        import torch

        import u32_prefix_scan_gb300 as u
        from u32_prefix_scan_gb300 import _native

        self.u = u
        self.keys = torch.from_numpy(host["keys"].view(np.int32)).to(dev)
        self.perm = None if self.mode == "keys" else torch.empty(self.n, dtype=torch.int32, device=dev)
        self.keys_out = None if self.mode == "perm" else torch.empty(self.n, dtype=torch.int32, device=dev)
        self.ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_RADIX, self.n), dev)
        self.pinned_in = {"keys": torch.from_numpy(host["keys"].view(np.int32)).pin_memory()}
        self.pinned_out = {}
        if self.perm is not None:
            self.pinned_out["perm"] = torch.empty(self.n, dtype=torch.int32).pin_memory()
        if self.keys_out is not None:
            self.pinned_out["keys_out"] = torch.empty(self.n, dtype=torch.int32).pin_memory()

    def step(self):
        if self.mode == "perm":
            self.u.radix_sort_perm_u32(self.keys, self.perm, workspace=self.ws)
        else:
            self.u.radix_sort_u32(self.keys, self.keys_out, self.perm, workspace=self.ws)

    def e2e_step(self):
        self.keys.copy_(self.pinned_in["keys"], non_blocking=True)
        self.step()
        for name, t in self.pinned_out.items():
            t.copy_(getattr(self, name), non_blocking=True)
        return 4 * self.n, 4 * self.n * len(self.pinned_out)

    def check_e2e(self, host):
        import numpy as np

        ok = True
        if "perm" in self.pinned_out:
            s = host["keys"][self.pinned_out["perm"].numpy()]
            ok &= bool(np.all(s[1:] >= s[:-1]))
        if "keys_out" in self.pinned_out:
            ok &= bool(np.array_equal(self.pinned_out["keys_out"].numpy().view(np.uint32), np.sort(host["keys"])))
        return ok

    def library_context(self, host, steps: int):
        """PyTorch's CUDA stable sort of the same keys, for context:
        torch.sort(stable=True) over int32 keys with the sign bit flipped
        (signed order of k ^ 2^31 is the unsigned order of k; the flip is
        done once, outside the timing) returns the sorted keys and int64
        indices, which are compared with this library's permutation."""
        import numpy as np
        import torch

        flipped = torch.from_numpy((host["keys"] ^ np.uint32(1 << 31)).view(np.int32)).to(self.keys.device)
        perm = torch.empty(self.n, dtype=torch.int32, device=self.keys.device)
        self.u.radix_sort_perm_u32(self.keys, perm, workspace=self.ws)
        _, idx = torch.sort(flipped, stable=True)
        torch.cuda.synchronize()
        same = bool(torch.equal(idx.to(torch.int32), perm))
        del perm, idx
        for _ in range(3):
            torch.sort(flipped, stable=True)
        stream = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(steps):
            torch.sort(flipped, stable=True)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        return {"call": "torch.sort(int32 keys ^ 2^31, stable=True) -> sorted keys + int64 indices, same device keys",
                "ms_per_step": ms, "value": self.n / (ms * 1e-3) / 1e9, "unit": UNIT,
                "indices_equal_to_radix_sort_perm_u32": same}

    def oracle_step(self, lib, arrays):
        import numpy as np

        k = arrays["keys"]
        if "perm" not in arrays:
            arrays["perm"] = np.empty(k.size, dtype=np.int32)
        lib.oracle_sort_perm_u32(k.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), k.size,
                                 arrays["perm"].ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
        if self.mode != "perm":
            arrays["keys_out"] = k[arrays["perm"]]


class RunsOp(Op):
    """The runs layout (in place) and the owner row. The layout replaces the
    counts by their ends, so every step first restores the counts with a
    device-to-device copy (part of the step's time, not of the kernels')."""

    log2n = 25
    launches_per_step = 3  # layout: scan + entries/slots fill; owner
    kernel_sources = ["u32_prefix_scan_gb300/csrc/runs.cu"]

    def __init__(self, args):
        super().__init__(args)
        self.skewed = args.skewed
        self.name = "runs_owner_u32" + ("_skewed" if self.skewed else "")
        mix = "skewed counts, 1/16 of owners in [0,64)" if self.skewed else "counts uniform in [0,8)"
        self.metric = f"runs layout + owner row Gelem/s (owners) at n=2^25 owners ({mix}), 1 GB300"
        self.kernel = "runs_owner_kernel<16 warps, 16 positions a lane> (merge path of ends with entry indices)"
        self.entries = None

    def workload(self):
        mix = "u32(6,0,i): d & 15 == 0 ? d >> 26 : 0" if self.skewed else "u32(6,0,i) >> 29"
        e = "" if self.entries is None else f", {self.entries} entries"
        return (f"runs of n=2^{self.n.bit_length() - 1} owners, counts {mix}{e}: ends in place + entries + "
                f"-1 slots, then owner(e) for every entry (counts restored by a device copy each step)")

    def algorithmic_bytes(self):
        # the owner kernel: ends read (4 per owner), owner row written (4 per entry)
        return 4 * self.n + 4 * self.entries

    def host_inputs(self):
        from u32_prefix_scan_gb300 import inputs

        c = inputs.run_counts(self.n, 6, skewed=self.skewed)
        self.entries = max(int(c.sum(dtype="u8")), 1)
        return {"counts": c}

    def setup(self, dev, host):
        import numpy as np
        import torch

        import u32_prefix_scan_gb300 as u
        from u32_prefix_scan_gb300 import _native

        self.u = u
        self.pristine = torch.from_numpy(host["counts"].view(np.int32)).to(dev)
        self.ends = torch.empty_like(self.pristine)
        self.entries_d = torch.empty(1, dtype=torch.int32, device=dev)
        self.slots = torch.empty(self.entries, dtype=torch.int32, device=dev)
        self.owner = torch.empty(self.entries, dtype=torch.int32, device=dev)
        self.ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_RUNS, self.n), dev)
        self.pinned_in = {"counts": torch.from_numpy(host["counts"].view(np.int32)).pin_memory()}
        self.pinned_out = {"ends": torch.empty(self.n, dtype=torch.int32).pin_memory(),
                           "entries": torch.empty(1, dtype=torch.int32).pin_memory(),
                           "owner": torch.empty(self.entries, dtype=torch.int32).pin_memory()}

    def _layout(self):
        self.u.runs_layout_u32(self.ends, self.entries_d, self.slots, workspace=self.ws)

    def _owner(self):
        self.u.runs_owner_u32(self.ends, self.owner, capacity=self.entries)

    def step(self):
        self.ends.copy_(self.pristine)
        self._layout()
        self._owner()

    def step_marked(self, before, after):
        self.ends.copy_(self.pristine)
        self._layout()
        before.record()
        self._owner()
        after.record()

    def e2e_step(self):
        self.ends.copy_(self.pinned_in["counts"], non_blocking=True)
        self._layout()
        self._owner()
        for name, t in (("ends", self.ends), ("entries", self.entries_d), ("owner", self.owner)):
            self.pinned_out[name].copy_(t, non_blocking=True)
        return 4 * self.n, 4 * self.n + 4 + 4 * self.entries

    def check_e2e(self, host):
        import numpy as np

        ends = self.pinned_out["ends"].numpy().view(np.uint32)
        if not np.array_equal(ends, np.cumsum(host["counts"], dtype=np.uint64).astype(np.uint32)):
            return False
        if int(self.pinned_out["entries"][0]) != self.entries:
            return False
        k = min(self.entries, 1 << 20)
        want = np.searchsorted(ends, np.arange(k, dtype=np.int64), side="right")
        return bool(np.array_equal(self.pinned_out["owner"][:k].numpy(), want))

    def oracle_step(self, lib, arrays):
        import numpy as np

        c = arrays["counts"]
        if "ends" not in arrays:
            arrays["ends"] = np.empty(c.size, dtype=np.uint32)
            arrays["slots"] = np.empty(max(int(c.sum(dtype="u8")), 1), dtype=np.int32)
        u32p, i32p = ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_int32)
        entries = lib.oracle_runs_layout_u32(c.ctypes.data_as(u32p), c.size, arrays["ends"].ctypes.data_as(u32p))
        lib.oracle_runs_fill_owner(c.ctypes.data_as(u32p), arrays["ends"].ctypes.data_as(u32p), c.size,
                                   arrays["slots"].ctypes.data_as(i32p), entries)


OPS = ["scan_exclusive", "scan_inclusive", "scan_op", "scan64", "segscan", "segscan_sums", "segreduce", "compact",
       "radix", "runs"]


def make_op(args) -> Op:
    if args.op in ("scan_exclusive", "scan_inclusive"):
        return ScanOp(args, args.op == "scan_inclusive")
    if args.op == "scan_op":
        return ScanOp(args, args.inclusive, args.monoid)
    if args.op == "compact":
        return CompactOp(args) if args.project == "indices" else CompactValuesOp(args)
    if args.op == "radix":
        return RadixOp(args)
    if args.op == "runs":
        return RunsOp(args)
    if args.op == "scan64":
        return Scan64Op(args)
    return SegOp(args, args.op)


# -------------------------------------------------------------- helpers ----

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--op", choices=OPS, default="scan_exclusive")
    p.add_argument("--heads", choices=["geometric", "regular4"], default="geometric")
    p.add_argument("--p", type=float, choices=[0.1, 0.9], default=0.1, help="compaction keep probability")
    p.add_argument("--ties", action="store_true", help="radix: keys in [0, 256) instead of uniform u32")
    p.add_argument("--sort", choices=["perm", "pairs", "keys"], default="perm",
                   help="radix outputs: the permutation, sorted keys and the permutation, or sorted keys only")
    p.add_argument("--project", choices=["indices", "values", "nonzero"], default="indices",
                   help="compact: kept indices (offsets, -1 tail), kept values by flags, or kept non-zero values")
    p.add_argument("--u8heads", action="store_true", help="segmented ops: one byte per head flag")
    p.add_argument("--monoid64", choices=["add", "mul", "and", "or", "xor", "min", "max"], default="add",
                   help="scan64: the operator")
    p.add_argument("--skewed", action="store_true", help="runs: the skewed count mix instead of uniform [0, 8)")
    p.add_argument("--monoid", choices=["add", "mul", "and", "or", "xor", "min", "max"], default="max",
                   help="scan_op: the operator")
    p.add_argument("--inclusive", action="store_true", help="scan_op: inclusive instead of exclusive")
    p.add_argument("--graph", action="store_true",
                   help="capture the timed steps in one CUDA graph and time its replay (launch-bound sizes)")
    p.add_argument("--library-context", action="store_true",
                   help="add scans / radix: also time torch.cumsum / torch.sort on the same inputs (context)")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--soak-seconds", type=float, default=1.0,
                   help="after the timed region, repeat timed windows of the same steps this long (clock record)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-rows", action="store_true",
                   help="default scan line: skip timing the other primitives on their workloads")
    p.add_argument("--log2n", type=int, default=None,
                   help="array size 2^log2n instead of the workload's (for profiler captures)")
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be at least 3")
    if a.steps < 1:
        p.error("--steps must be at least 1")
    return a


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def source_hash(rels) -> str:
    h = hashlib.sha256()
    for rel in rels:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def load_peak():
    f = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(f.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def host_cpu() -> str:
    """The host CPU's model name (context for the CPU baseline)."""
    try:
        for line in open("/proc/cpuinfo"):
            key, _, val = line.partition(":")
            if key.strip() in ("model name", "CPU part", "Model"):
                return val.strip()
    except OSError:
        pass
    import platform

    return platform.machine()


def copy_peak_gbs(dev, nbytes: int = 1 << 30, reps: int = 20) -> float:
    """Device-to-device copy bandwidth measured now, on this GPU: read +
    write bytes of `reps` copies of a 1 GiB buffer over their event time."""
    import torch

    a = torch.empty(nbytes // 4, dtype=torch.int32, device=dev)
    b = torch.empty_like(a)
    a.fill_(1)
    for _ in range(3):
        b.copy_(a)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        b.copy_(a)
    e1.record()
    torch.cuda.synchronize()
    gbs = 2 * nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del a, b
    return gbs


def load_traffic(op: Op):
    """ncu DRAM bytes per launch, if captured for the current kernel source
    at this workload size."""
    try:
        d = json.loads(op.traffic_file.read_text())
    except Exception:
        return None
    if d.get("source_hash") != source_hash(op.kernel_sources) or d.get("scaled_to_n") != op.n:
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

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock, its maximum and the throttle reasons seen in
        [t0, t1] (the samples around it when none fall inside)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = [l for (t, l) in self.lines if t0 is None or (t0 - 0.06 <= t <= t1 + 0.06)]
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


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def time_oracle(op: Op, host: dict, seconds: float, sample: int):
    """The oracle (one thread, as it stands) repeated on the first `sample`
    elements of the workload until `seconds` pass. Returns elements/s."""
    import oracle

    lib = oracle._load()
    arrays = {k: v[:sample].copy() for k, v in host.items()}
    reps, t0 = 0, time.perf_counter()
    while True:
        op.oracle_step(lib, arrays)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return sample * reps / el, reps, el


# ----------------------------------------------------------------- arms ----

def run_reference(args, rank):
    """The reference arm: the CPU oracle on the host cores, rank 0 only."""
    if rank != 0:
        return None
    import oracle

    oracle.build()
    op = make_op(args)
    host = op.host_inputs()
    sample = min(op.n, REF_SAMPLE)
    lib = oracle._load()
    arrays = {k: v[:sample].copy() for k, v in host.items()}
    for _ in range(args.warmup):
        op.oracle_step(lib, arrays)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        op.oracle_step(lib, arrays)
    el = time.perf_counter() - t0
    value = sample * args.steps / el / 1e9
    desc = f"{op.name} oracle on the first 2^{sample.bit_length() - 1} elements of the workload per step"
    return {
        "impl": "reference", "metric": op.metric, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": op.workload(), "n": op.n, "op": args.op, "sample_per_step": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc,
                         "host_cpu": host_cpu(), "host_nproc": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def measure_host_link(op, stream, reps: int = 3):
    """The host link's copy rates in this run (GB/s): host to device, device
    to host, and both at once on two streams, with the step's own page-locked
    buffers (the largest input and output) and a device buffer of the same
    size; the best of `reps` each. None when the step has no such buffers."""
    import torch

    ins = [t for t in getattr(op, "pinned_in", {}).values() if t.numel() > 1]
    outs = [t for t in getattr(op, "pinned_out", {}).values() if t.numel() > 1]
    if not ins or not outs:
        return None
    h_in = max(ins, key=lambda t: t.numel() * t.element_size()).view(torch.uint8)
    h_out = max(outs, key=lambda t: t.numel() * t.element_size()).view(torch.uint8)
    nbytes = min(h_in.numel(), h_out.numel())
    h_in, h_out = h_in[:nbytes], h_out[:nbytes]
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=stream.device)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=stream.device)
    s1, s2 = torch.cuda.Stream(stream.device), torch.cuda.Stream(stream.device)

    def timed(fn):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None or ms < best else best
        return best

    def both():
        s1.wait_stream(stream)
        s2.wait_stream(stream)
        with torch.cuda.stream(s1):
            d_a.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_b, non_blocking=True)
        stream.wait_stream(s1)
        stream.wait_stream(s2)

    with torch.cuda.stream(stream):
        h2d = timed(lambda: d_a.copy_(h_in, non_blocking=True))
        d2h = timed(lambda: h_out.copy_(d_b, non_blocking=True))
        two = timed(both)
    del d_a, d_b
    return {"h2d": nbytes / (h2d * 1e-3) / 1e9, "d2h": nbytes / (d2h * 1e-3) / 1e9,
            "both": 2 * nbytes / (two * 1e-3) / 1e9, "bytes_each_way": nbytes}


def parse_cpulist(text: str) -> set:
    """CPUs of a sysfs cpulist such as "0-15,32-47"."""
    cpus = set()
    for part in text.strip().split(","):
        if part:
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
    return cpus


def bind_to_gpu_numa_node(dev_index: int):
    """Bind this process to the CPUs of the GPU's NUMA node, so that the
    page-locked host buffers of the end-to-end leg are allocated next to the
    GPU's host link. Returns the node, or None when sysfs does not name one
    (the affinity is then left as it was)."""
    import torch

    try:
        p = torch.cuda.get_device_properties(dev_index)
        addr = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        node = int(pathlib.Path(f"/sys/bus/pci/devices/{addr}/numa_node").read_text())
        if node < 0:
            return None
        cpus = parse_cpulist(pathlib.Path(f"/sys/devices/system/node/node{node}/cpulist").read_text())
        mine = os.sched_getaffinity(0) & cpus
        if mine:
            os.sched_setaffinity(0, mine)
            return node
    except (AttributeError, OSError, ValueError):
        pass
    return None


ROW_WORKLOADS = [
    ["--op", "segscan"],
    ["--op", "segscan_sums"],
    ["--op", "segscan_sums", "--heads", "regular4"],
    ["--op", "segreduce"],
    ["--op", "segreduce", "--heads", "regular4"],
    ["--op", "compact"],
    ["--op", "compact", "--p", "0.9"],
    ["--op", "radix"],
    ["--op", "radix", "--ties"],
]


def measure_rows(dev, stream, peak: float, seconds: float = 0.3):
    """The other primitives on their own workloads, each timed on the device
    like the headline (warm-up, then a timed run of about `seconds`, events
    on the launching stream), so that one bench line carries every
    primitive's fraction of the copy peak."""
    import torch

    rows = []
    sampler = ClockSampler(torch.cuda.current_device()).start()
    t_start = time.time()
    for argv in ROW_WORKLOADS:
        a = parse_args(argv)
        a.world, a.rank = 1, 0
        op = make_op(a)
        op.setup(dev, op.host_inputs())
        marked = op.is_marked()
        for _ in range(5):
            op.step()
        torch.cuda.synchronize()
        t0 = time.time()
        for _ in range(5):
            op.step()
        torch.cuda.synchronize()
        steps = max(50, int(seconds / max((time.time() - t0) / 5, 1e-6)))
        marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(steps if marked else 0)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(steps):
            if marked:
                op.step_marked(*marks[k])
            else:
                op.step()
        end.record(stream)
        torch.cuda.synchronize()
        op.u.check(workspace=op.ws)
        ms = start.elapsed_time(end) / steps
        kernel_ms = sum(x.elapsed_time(y) for x, y in marks) / steps if marked else ms
        achieved = op.algorithmic_bytes() / (kernel_ms * 1e-3) / 1e9
        rows.append({"op": " ".join(argv[1:]), "workload": op.workload(), "value": op.n / (ms * 1e-3) / 1e9,
                     "unit": UNIT, "steps": steps, "ms_per_step": ms, "hbm_gbs": achieved, "frac": achieved / peak,
                     "algorithmic_bytes_per_step": op.algorithmic_bytes(), "traffic": load_traffic(op)})
        del op, marks
        torch.cuda.empty_cache()
    sampler.stop()
    return {"note": "each primitive timed on the device in this run, L2 not flushed (inputs above 129 MB); "
                    "frac is of the measured copy peak",
            "clocks": sampler.summary(t_start, time.time()), "rows": rows}


def run_ours(args, rank, local_rank, world):
    import torch

    from u32_prefix_scan_gb300 import build as native_build

    native_build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    numa_node = bind_to_gpu_numa_node(local_rank)  # before any host buffer is pinned
    stream = torch.cuda.current_stream()
    args.world, args.rank = world, rank
    op = make_op(args)
    host = op.host_inputs()
    op.setup(dev, host)

    for _ in range(args.warmup):
        op.step()
    op.u.check(workspace=op.ws)

    sampler = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.15)
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # an op whose step runs several calls brackets its dominant kernel with
    # events on the launching stream; the roofline uses that kernel's time
    marked = op.is_marked()
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps if marked else 0)]
    graph = None
    if args.graph:
        # the K timed steps captured once, replayed once inside the timed
        # region: no host launch cost between steps (for L2-resident sizes,
        # where the host's launch rate would otherwise be what is timed)
        if marked:
            raise SystemExit("bench: --graph times plain steps; this op brackets its dominant kernel with events")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                op.step()
        graph.replay()  # one untimed replay
        torch.cuda.synchronize()
    w0 = time.time()
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for k in range(args.steps):
            if marked:
                op.step_marked(*marks[k])
            else:
                op.step()
    end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    # Repeat windows of the same K steps for about --soak-seconds (timed
    # each, reported apart from the timed region), so that the clock record
    # holds more than the few samples a short timed region gets.
    soak = []
    w2 = time.time()
    while args.soak_seconds > 0 and time.time() - w2 < args.soak_seconds:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for k in range(args.steps):
                op.step()
        b.record(stream)
        torch.cuda.synchronize()
        soak.append(a.elapsed_time(b) / args.steps)
    w3 = time.time()
    barrier(world)
    sampler.stop()
    clocks = sampler.summary(w0, w1)
    op.u.check(workspace=op.ws)
    ms = start.elapsed_time(end) / args.steps
    ms_max = max_over_ranks(ms, world)
    kernel_ms = sum(a.elapsed_time(b) for a, b in marks) / args.steps if marked else ms

    # end to end through the C ABI: pinned host inputs in, outputs back out
    h2d = d2h = 0
    e2e_ms = None
    link = None
    if args.e2e_steps:
        for _ in range(2):
            op.e2e_step()
        torch.cuda.synchronize()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        for _ in range(args.e2e_steps):
            h2d, d2h = op.e2e_step()
        e_end.record(stream)
        torch.cuda.synchronize()
        op.u.check(workspace=op.ws)
        if getattr(op, "ws_host", None) is not None:
            op.u.check(workspace=op.ws_host)
        e2e_ms = max_over_ranks(e_start.elapsed_time(e_end) / args.e2e_steps, world)
        if not op.check_e2e(host):
            raise SystemExit("bench: e2e result fails its property check")
        link = measure_host_link(op, stream)

    library = None
    if args.library_context:
        if not hasattr(op, "library_context") or getattr(op, "monoid", "add") != "add":
            raise SystemExit("bench: --library-context applies to the U32 add scans and the radix sort")
        library = op.library_context(host, args.steps)

    peak, peak_kind = load_peak()
    nbytes = op.algorithmic_bytes()
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    copy_now = copy_peak_gbs(dev)
    full = op.n == 1 << op.log2n
    result = {
        "metric": op.metric,
        "value": world * op.n / (ms_max * 1e-3) / 1e9,
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
        "config": {"workload": op.workload() if full else f"profiling case: {op.workload()}", "n": op.n,
                   "op": args.op, "per_rank": "one independent replica per GPU",
                   "l2": ("inputs larger than the 129 MB L2; no flush between steps" if nbytes > L2_BYTES
                          else "inputs resident in the 129 MB L2: a latency figure, no roofline claim"),
                   **({"launch": "the timed steps replayed from one CUDA graph"} if graph is not None else {})},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": load_traffic(op), "algorithmic_bytes_per_launch": nbytes, "kernel": op.kernel,
                     "kernel_ms": kernel_ms, "copy_gbs_same_run": copy_now, "frac_of_same_run_copy": achieved / copy_now,
                     "nominal_gbs": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS},
        "e2e": {"value": world * op.n / (e2e_ms * 1e-3) / 1e9 if e2e_ms else None, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "host_numa_node": numa_node,
                "host_link_gbs": link,
                "frac_of_host_link": ((h2d + d2h) / (e2e_ms * 1e-3) / 1e9 / link["both"]) if link and e2e_ms else None},
        "clocks": clocks,
        "gpu_launches": args.steps * op.launches_per_step,
    }
    if soak:
        soak.sort()
        result["repeat_windows"] = {"windows": len(soak), "steps_each": args.steps,
                                    "ms_per_step_median": soak[len(soak) // 2], "ms_per_step_min": soak[0],
                                    "ms_per_step_max": soak[-1], "clocks": sampler.summary(w2, w3)}
    if getattr(op, "sharded", False):
        result["scaling"] = "weak"
        result["config"]["per_rank"] = (
            f"one shard of one global compaction: count (4 B/elem), all-gather of the {world} (count, length) "
            "pairs over NCCL, compaction from the carry-ins (12 B/elem)" if isinstance(op, CompactOp) else
            f"one shard of one global segmented scan: its own scan (12 B/elem), all-gather of the {world} "
            "(head, tail, count) summaries over NCCL, the carry-in added before its first head"
            if isinstance(op, SegOp) else
            "one shard of one global scan: fold (4 B/elem), all-gather of the "
            f"{world} shard sums over NCCL, scan from the carry-in (8 B/elem)")
    if library is not None:
        if "hbm_gbs" in library:
            library["frac"] = library["hbm_gbs"] / peak
        result["library_context"] = library
    if world == 1 and args.op == "scan_exclusive" and args.log2n is None and not args.no_rows:
        result["other_rows"] = measure_rows(dev, stream, peak)
    if rank == 0 and not args.no_cpu_baseline:
        v, reps, el = time_oracle(op, host, args.cpu_seconds, op.n)
        result["cpu_baseline"] = {"value": v / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
                                  "host_cpu": host_cpu(), "host_nproc": os.cpu_count(),
                                  "sample": f"{op.name} oracle over the full workload "
                                            f"(n=2^{op.n.bit_length() - 1}), {reps} repetitions in {el:.1f} s"}
    return result


def main(argv=None):
    args = parse_args(argv)
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        # rank 0 alone times the oracle; other ranks exit without work
        out = run_reference(args, rank)
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

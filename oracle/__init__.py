"""CPU oracle for the U32 scan primitives (numpy front end over oracle.c).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
CPU-baseline / reference legs may import this package. The CUDA library and
its Python binding never import it, and it imports nothing from them: the two
share no code. Inputs come from the seeded generator module, passed in as
arrays.

Every wrapper copies its inputs, calls one plain sequential C function
(oracle.c, one thread) and returns new arrays; see oracle.c for the passage
of the source pages each function follows. Nothing here is tuned.

Parity pins: every function is pinned in tests/test_oracle_pins.py against
values the pages print (tests/golden/), closed forms, invariants the pages
state, independent library routines (numpy) and brute force on tiny inputs.
"""

from __future__ import annotations

import ctypes
import os
import pathlib
import subprocess

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_SO = _HERE / "liboracle.so"

_u32p = ctypes.POINTER(ctypes.c_uint32)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u64 = ctypes.c_uint64

_lib = None


def build(force: bool = False) -> pathlib.Path:
    """Compile oracle.c into liboracle.so (plain gcc -O2, no target flags)."""
    if force or not _SO.exists() or _SO.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _SO.with_suffix(f".so.tmp{os.getpid()}")
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC",
             "-o", str(tmp), str(_SRC)])
        os.replace(tmp, _SO)
    return _SO


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    lib.oracle_scan_exclusive_u32.argtypes = [_u32p, _u64]
    lib.oracle_scan_exclusive_u32.restype = ctypes.c_uint32
    lib.oracle_scan_inclusive_u32.argtypes = [_u32p, _u64]
    lib.oracle_scan_inclusive_u32.restype = ctypes.c_uint32
    lib.oracle_scan_op_u32.argtypes = [ctypes.c_int, ctypes.c_int, _u32p, _u64]
    lib.oracle_scan_op_u32.restype = ctypes.c_uint32
    lib.oracle_scan_blocked_u32.argtypes = [ctypes.c_int, ctypes.c_uint, _u32p, _u64, _u32p]
    lib.oracle_scan_blocked_u32.restype = ctypes.c_uint32
    lib.oracle_segscan_inclusive_u32.argtypes = [_u32p, _i32p, _u64]
    lib.oracle_segscan_inclusive_u32.restype = None
    lib.oracle_segreduce_u32.argtypes = [_u32p, _i32p, _u64, _u32p]
    lib.oracle_segreduce_u32.restype = ctypes.c_uint64
    lib.oracle_compact_indices.argtypes = [_i32p, _u64, _i32p, _i32p, _i32p]
    lib.oracle_compact_indices.restype = ctypes.c_int32
    lib.oracle_radix_perm_bits.argtypes = [_u32p, _u64, ctypes.c_uint, _i32p, _i32p, _i32p]
    lib.oracle_radix_perm_bits.restype = None
    lib.oracle_sort_perm_u32.argtypes = [_u32p, _u64, _i32p]
    lib.oracle_sort_perm_u32.restype = ctypes.c_int
    lib.oracle_runs_layout_u32.argtypes = [_u32p, _u64, _u32p]
    lib.oracle_runs_layout_u32.restype = ctypes.c_uint32
    lib.oracle_runs_fill_owner.argtypes = [_u32p, _u32p, _u64, _i32p, _u64]
    lib.oracle_runs_fill_owner.restype = None
    lib.oracle_compact_values_u32.argtypes = [_u32p, _i32p, _u64, _u32p]
    lib.oracle_compact_values_u32.restype = ctypes.c_uint64
    lib.oracle_scan_op_u64.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64), _u64]
    lib.oracle_scan_op_u64.restype = ctypes.c_uint64
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(str(build())))
    return _lib


def _u32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint32:
        if a.size and (a.min() < 0 or a.max() >= (1 << 32)):
            raise ValueError("values must lie in [0, 2^32)")
        a = a.astype(np.uint32)
    return np.ascontiguousarray(a).copy()


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32)).copy()


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def scan_exclusive(a):
    """(scanned copy, total): out[j] = a[0] + .. + a[j-1] mod 2^32."""
    out = _u32(a)
    total = _load().oracle_scan_exclusive_u32(_p(out, _u32p), out.size)
    return out, int(total)


def scan_inclusive(a):
    """(scanned copy, total): out[j] = a[0] + .. + a[j] mod 2^32."""
    out = _u32(a)
    total = _load().oracle_scan_inclusive_u32(_p(out, _u32p), out.size)
    return out, int(total)


SCAN_OPS = {"add": 0, "mul": 1, "and": 2, "or": 3, "xor": 4, "min": 5, "max": 6}


def scan_op(a, op: str, inclusive: bool):
    """(scanned copy, fold) under one of the CAIRN integer operators on
    uint32: add, mul (both wrapping), and, or, xor, min, max."""
    out = _u32(a)
    total = _load().oracle_scan_op_u32(SCAN_OPS[op], int(bool(inclusive)), _p(out, _u32p), out.size)
    return out, int(total)


def scan_blocked(a, b: int, inclusive: bool):
    """The three-pass blocked scan at fork depth b: (scanned copy, total)."""
    out = _u32(a)
    d = min(int(b), 30, max(out.size, 1).bit_length() - 1)
    scratch = np.zeros(1 << d, dtype=np.uint32)
    total = _load().oracle_scan_blocked_u32(int(bool(inclusive)), int(b), _p(out, _u32p),
                                            out.size, _p(scratch, _u32p))
    return out, int(total)


def segscan_inclusive(a, flags):
    """Segmented inclusive scan (copy); a non-zero flag opens a segment."""
    out = _u32(a)
    f = _i32(flags)
    if f.size != out.size:
        raise ValueError("values and flags differ in length")
    _load().oracle_segscan_inclusive_u32(_p(out, _u32p), _p(f, _i32p), out.size)
    return out


def segreduce(a, flags):
    """(per-segment wrapped sums in segment order, number of segments)."""
    v = _u32(a)
    f = _i32(flags)
    if f.size != v.size:
        raise ValueError("values and flags differ in length")
    sums = np.zeros(max(v.size, 1), dtype=np.uint32)
    nseg = _load().oracle_segreduce_u32(_p(v, _u32p), _p(f, _i32p), v.size, _p(sums, _u32p))
    return sums[:nseg].copy(), int(nseg)


def compact_indices(flags):
    """(inclusive offsets, indices with a -1 tail, count)."""
    f = _i32(flags)
    n = f.size
    if n >= (1 << 31):
        raise ValueError("n must be below 2^31")
    offsets = np.empty(n, dtype=np.int32)
    indices = np.empty(n, dtype=np.int32)
    count = np.zeros(1, dtype=np.int32)
    _load().oracle_compact_indices(_p(f, _i32p), n, _p(offsets, _i32p), _p(indices, _i32p),
                                   _p(count, _i32p))
    return offsets, indices, int(count[0])


def radix_perm_bits(keys, bits: int = 32):
    """The sort graph's permutation: LSD, one bit per pass, `bits` passes."""
    k = _u32(keys)
    n = k.size
    if n >= (1 << 31):
        raise ValueError("n must be below 2^31")
    if not 1 <= bits <= 32:
        raise ValueError("bits must be in 1..32")
    perm = np.empty(n, dtype=np.int32)
    zeros = np.empty(n, dtype=np.int32)
    slots = np.empty(n, dtype=np.int32)
    _load().oracle_radix_perm_bits(_p(k, _u32p), n, bits, _p(perm, _i32p), _p(zeros, _i32p),
                                   _p(slots, _i32p))
    return perm


def sort_perm(keys):
    """The unique stable sorting permutation, by (key, index) order."""
    k = _u32(keys)
    n = k.size
    if n >= (1 << 31):
        raise ValueError("n must be below 2^31")
    perm = np.empty(n, dtype=np.int32)
    if _load().oracle_sort_perm_u32(_p(k, _u32p), n, _p(perm, _i32p)) != 0:
        raise MemoryError("oracle_sort_perm_u32 could not allocate")
    return perm


def runs_layout(counts):
    """(ends, entries): ends the inclusive scan of the counts (mod 2^32),
    entries = max(total, 1)."""
    c = _u32(counts)
    ends = np.empty(c.size, dtype=np.uint32)
    entries = _load().oracle_runs_layout_u32(_p(c, _u32p), c.size, _p(ends, _u32p))
    return ends, int(entries)


def runs_owner(counts):
    """(ends, entries, owner row): the runs layout, then its `entries` slots
    filled by the scatter over the owners with each owner's index, so that
    slot e holds owner(e, ends); -1 where no run reaches."""
    c = _u32(counts)
    if c.size >= (1 << 31):
        raise ValueError("n must be below 2^31")
    ends, entries = runs_layout(c)
    slots = np.empty(entries, dtype=np.int32)
    _load().oracle_runs_fill_owner(_p(c, _u32p), _p(ends, _u32p), c.size, _p(slots, _i32p), entries)
    return ends, entries, slots


def compact_values(values, flags=None, out=None):
    """(out, count): the kept values in order at the front of a copy of
    `out` (zeros when not given), the rest of it unchanged. An element is
    kept when its flag is non-zero, or, with no flags, its value is."""
    v = _u32(values)
    o = np.zeros(v.size, dtype=np.uint32) if out is None else _u32(out)
    if o.size != v.size:
        raise ValueError("out must have n elements")
    f = None if flags is None else _i32(flags)
    if f is not None and f.size != v.size:
        raise ValueError("values and flags differ in length")
    used = _load().oracle_compact_values_u32(_p(v, _u32p), None if f is None else _p(f, _i32p), v.size,
                                            _p(o, _u32p))
    return o, int(used)


def scan_op_u64(a, op: str, inclusive: bool):
    """(scanned copy, fold) of a uint64 row under one of the CAIRN integer
    operators (add and mul wrap at 2^64)."""
    out = np.ascontiguousarray(np.asarray(a, dtype=np.uint64)).copy()
    total = _load().oracle_scan_op_u64(SCAN_OPS[op], int(bool(inclusive)),
                                       out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), out.size)
    return out, int(total)

"""ctypes view of libu32scan.so: the C ABI declared in include/u32scan.h.

Loading fails loudly when the library has not been built; there is no
fallback implementation anywhere in this package.
"""

from __future__ import annotations

import ctypes
import pathlib

SO = pathlib.Path(__file__).resolve().parent / "libu32scan.so"

OK = 0
EINVAL = -1
EWORKSPACE = -2
ECUDA = -3
ETIMEOUT = -4

SCAN_OPS = {"add": 0, "mul": 1, "and": 2, "or": 3, "xor": 4, "min": 5, "max": 6}

OP_SCAN = 1
OP_SEGSCAN = 2
OP_COMPACT = 3
OP_RADIX = 4
OP_RUNS = 5
OP_SCAN64 = 6
OP_SCAN_HOST = 7
OP_REDUCE = 8

_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_int = ctypes.c_int

# name -> (restype, argtypes)
SIGNATURES = {
    "u32scan_workspace_bytes": (_sz, [_int, _sz]),
    "u32scan_workspace_init": (_int, [_vp, _sz, _vp]),
    "u32scan_check": (_int, [_vp, _vp]),
    "u32scan_strerror": (ctypes.c_char_p, [_int]),
    "u32scan_version": (_int, []),
    "scan_exclusive_u32": (_int, [_vp, _sz, _vp, _vp, _sz, _vp]),
    "scan_inclusive_u32": (_int, [_vp, _sz, _vp, _vp, _sz, _vp]),
    "scan_exclusive_u32_noalloc": (_int, [_vp, _sz, _vp, _vp]),
    "scan_exclusive_u32_carry": (_int, [_vp, _sz, _vp, _vp, _vp, _sz, _vp]),
    "scan_inclusive_u32_carry": (_int, [_vp, _sz, _vp, _vp, _vp, _sz, _vp]),
    "reduce_u32_op": (_int, [_int, _vp, _sz, _vp, _vp, _sz, _vp]),
    "count_nonzero_u32": (_int, [_vp, _sz, _vp, _vp, _sz, _vp]),
    "u32scan_fill_splitmix_u32": (_int, [_vp, _sz, ctypes.c_uint, ctypes.c_uint, _sz, _vp]),
    "segscan_piece_summary_u32": (_int, [_vp, _vp, _sz, _vp, _int, _vp, _vp]),
    "segscan_piece_carries_u32": (_int, [_vp, _sz, _vp, _vp, _vp]),
    "segscan_fix_u32": (_int, [_vp, _vp, _sz, _vp, _vp, _sz, _vp]),
    "compact_indices_u32_carry": (_int, [_vp, _sz, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "scan_exclusive_u32_host": (_int, [_vp, _vp, _sz, _vp, _vp, _sz, _vp]),
    "scan_inclusive_u32_host": (_int, [_vp, _vp, _sz, _vp, _vp, _sz, _vp]),
    "scan_u32_op": (_int, [_int, _int, _vp, _sz, _vp, _vp, _sz, _vp]),
    "scan_u64_op": (_int, [_int, _int, _vp, _sz, _vp, _vp, _sz, _vp]),
    "segscan_inclusive_u32": (_int, [_vp, _vp, _sz, _vp, _sz, _vp, _vp, _sz, _vp]),
    "segreduce_u32": (_int, [_vp, _vp, _sz, _vp, _sz, _vp, _vp, _sz, _vp]),
    "segscan_inclusive_u32_u8heads": (_int, [_vp, _vp, _sz, _vp, _sz, _vp, _vp, _sz, _vp]),
    "segreduce_u32_u8heads": (_int, [_vp, _vp, _sz, _vp, _sz, _vp, _vp, _sz, _vp]),
    "compact_indices_u32": (_int, [_vp, _sz, _vp, _vp, _vp, _vp, _sz, _vp]),
    "compact_values_u32": (_int, [_vp, _vp, _sz, _vp, _vp, _vp, _sz, _vp]),
    "radix_sort_perm_u32": (_int, [_vp, _sz, _vp, _vp, _sz, _vp]),
    "radix_sort_u32": (_int, [_vp, _sz, _vp, _vp, _vp, _sz, _vp]),
    "runs_layout_u32": (_int, [_vp, _sz, _vp, _vp, _sz, _vp, _sz, _vp]),
    "runs_owner_u32": (_int, [_vp, _sz, _vp, _sz, _vp]),
    "u32scan_test_scan_skip_publish": (_int, [_vp, _sz, _vp, _vp, _sz, ctypes.c_uint, ctypes.c_ulonglong, _vp]),
    "u32scan_test_segscan_skip_publish": (_int, [_vp, _vp, _sz, _vp, _sz, _vp, _vp, _sz, ctypes.c_uint,
                                                  ctypes.c_ulonglong, _vp]),
    "u32scan_check_noalloc": (_int, [_vp]),
    "u32scan_test_noalloc_skip_publish": (_int, [_vp, _sz, _vp, ctypes.c_uint, ctypes.c_ulonglong, _vp]),
    "u32scan_test_noalloc_set_epoch": (_int, [ctypes.c_uint, _vp]),
}

_lib = None


class U32ScanError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} (status {status})")


def load(path) -> ctypes.CDLL:
    """A library built from these sources at `path` (e.g. with other launch
    shapes), with the same signatures declared."""
    handle = ctypes.CDLL(str(path))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib() -> ctypes.CDLL:
    """The loaded library with its signatures declared."""
    global _lib
    if _lib is None:
        if not SO.exists():
            raise RuntimeError(
                f"{SO.name} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                "(needs nvcc); this package has no CPU fallback")
        _lib = load(SO)
    return _lib


def strerror(status: int) -> str:
    return lib().u32scan_strerror(status).decode()


def check(status: int, what: str) -> None:
    if status != OK:
        raise U32ScanError(status, what)

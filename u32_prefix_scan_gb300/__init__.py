"""u32_prefix_scan_gb300: U32 prefix scans and the primitives built on them,
as hand-written CUDA kernels for GB300 (sm_103a) behind a C ABI
(include/u32scan.h, libu32scan.so), with a thin torch-tensor binding.

The tensor-level functions live in `api` (imported lazily so that the seeded
input generator in `inputs` can be used without torch or the library).
"""

_API = {
    "Workspace",
    "scan_exclusive_u32",
    "scan_inclusive_u32",
    "scan_exclusive_u32_carry",
    "scan_inclusive_u32_carry",
    "reduce_u32_op",
    "count_nonzero_u32",
    "fill_splitmix_u32",
    "segscan_piece_summary_u32",
    "segscan_piece_carries_u32",
    "segscan_fix_u32",
    "compact_indices_u32_carry",
    "scan_exclusive_u32_host",
    "scan_inclusive_u32_host",
    "scan_u32_op",
    "scan_u64_op",
    "segscan_inclusive_u32",
    "segreduce_u32",
    "compact_indices_u32",
    "compact_values_u32",
    "radix_sort_perm_u32",
    "radix_sort_u32",
    "runs_layout_u32",
    "runs_owner_u32",
    "check",
}


def __getattr__(name):
    if name in _API:
        from . import api

        return getattr(api, name)
    raise AttributeError(name)

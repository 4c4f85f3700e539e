"""Torch-tensor front end of libu32scan.so: argument marshalling only.

Every function takes CUDA tensors, checks dtype/device/contiguity, and
passes raw device pointers, sizes and the current CUDA stream to the C
entry point of the same name. All computation happens in the library's
kernels; nothing here touches tensor data.

U32 arrays are accepted as torch.int32 or torch.uint32 tensors (the bits are
the same; wrapping u32 addition and two's-complement int32 addition agree).
"""

from __future__ import annotations

import threading

import torch

from . import _native

__all__ = [
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
]

_U32_DTYPES = (torch.int32, getattr(torch, "uint32", torch.int32))


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _require_cuda(t: torch.Tensor, name: str, dtypes=_U32_DTYPES) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class Workspace:
    """Device workspace for the library's carries, reused across calls.

    One zero-filled byte buffer per (device, stream), grown on demand. The
    library keeps it consistent between calls by itself; calls sharing a
    workspace must be ordered, which one stream guarantees.
    """

    _lock = threading.Lock()
    _cache: dict = {}

    def __init__(self, nbytes: int, device: torch.device):
        self.buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def nbytes(self) -> int:
        return self.buf.numel()

    @classmethod
    def get(cls, op: int, n: int, device: torch.device, stream_handle: int) -> "Workspace":
        need = _native.lib().u32scan_workspace_bytes(op, n)
        key = (device.index, stream_handle)
        with cls._lock:
            ws = cls._cache.get(key)
            if ws is None or ws.nbytes < need:
                ws = cls(max(need, 2 * ws.nbytes if ws else need), device)
                cls._cache[key] = ws
        return ws


def _ws(op: int, n: int, device, stream_handle: int, workspace) -> Workspace:
    if workspace is not None:
        return workspace
    return Workspace.get(op, n, device, stream_handle)


def _scalar_out(out, like: torch.Tensor, dtype) -> torch.Tensor:
    if out is None:
        return torch.empty(1, dtype=dtype, device=like.device)
    _require_cuda(out, "out", (dtype,) if dtype not in _U32_DTYPES else _U32_DTYPES)
    if out.numel() < 1:
        raise ValueError("out must hold at least one element")
    return out


def _scan(name: str, data: torch.Tensor, total, stream, workspace) -> torch.Tensor:
    _require_cuda(data, "data")
    total = _scalar_out(total, data, data.dtype)
    n = data.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_SCAN, n, data.device, sh, workspace)
    fn = getattr(_native.lib(), name)
    _native.check(fn(data.data_ptr(), n, total.data_ptr(), ws.ptr, ws.nbytes, sh), name)
    return total


def scan_exclusive_u32(data: torch.Tensor, total: torch.Tensor | None = None, *, stream=None,
                       workspace: Workspace | None = None) -> torch.Tensor:
    """In place: data[j] <- data[0] + .. + data[j-1] (mod 2^32). Returns the
    one-element device tensor holding the wrapped total."""
    return _scan("scan_exclusive_u32", data, total, stream, workspace)


def scan_inclusive_u32(data: torch.Tensor, total: torch.Tensor | None = None, *, stream=None,
                       workspace: Workspace | None = None) -> torch.Tensor:
    """In place: data[j] <- data[0] + .. + data[j] (mod 2^32). Returns the
    one-element device tensor holding the wrapped total."""
    return _scan("scan_inclusive_u32", data, total, stream, workspace)


def _scan_carry(name: str, data: torch.Tensor, carry_in, total, stream, workspace) -> torch.Tensor:
    _require_cuda(data, "data")
    if carry_in is not None:
        _require_cuda(carry_in, "carry_in")
        if carry_in.numel() < 1:
            raise ValueError("carry_in must hold at least one element")
    total = _scalar_out(total, data, data.dtype)
    n = data.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_SCAN, n, data.device, sh, workspace)
    fn = getattr(_native.lib(), name)
    _native.check(fn(data.data_ptr(), n, carry_in.data_ptr() if carry_in is not None else None, total.data_ptr(),
                     ws.ptr, ws.nbytes, sh), name)
    return total


def scan_exclusive_u32_carry(data: torch.Tensor, carry_in: torch.Tensor | None, total: torch.Tensor | None = None,
                             *, stream=None, workspace: Workspace | None = None) -> torch.Tensor:
    """In place: data[j] <- carry_in + data[0] + .. + data[j-1] (mod 2^32),
    carry_in a one-element device tensor (None: 0). Returns the one-element
    device tensor holding carry_in + the wrapped sum of data."""
    return _scan_carry("scan_exclusive_u32_carry", data, carry_in, total, stream, workspace)


def scan_inclusive_u32_carry(data: torch.Tensor, carry_in: torch.Tensor | None, total: torch.Tensor | None = None,
                             *, stream=None, workspace: Workspace | None = None) -> torch.Tensor:
    """In place: data[j] <- carry_in + data[0] + .. + data[j] (mod 2^32).
    Returns carry_in + the wrapped sum of data (one-element device tensor)."""
    return _scan_carry("scan_inclusive_u32_carry", data, carry_in, total, stream, workspace)


def reduce_u32_op(data: torch.Tensor, op: str = "add", total: torch.Tensor | None = None, *, stream=None,
                  workspace: Workspace | None = None) -> torch.Tensor:
    """The fold of data under op in {add, mul, and, or, xor, min, max} (u32;
    add and mul wrap), read once. Returns a one-element device tensor."""
    if op not in _native.SCAN_OPS:
        raise ValueError(f"op must be one of {sorted(_native.SCAN_OPS)}")
    _require_cuda(data, "data")
    total = _scalar_out(total, data, data.dtype)
    n = data.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_REDUCE, n, data.device, sh, workspace)
    _native.check(_native.lib().reduce_u32_op(_native.SCAN_OPS[op], data.data_ptr(), n, total.data_ptr(), ws.ptr,
                                              ws.nbytes, sh), "reduce_u32_op")
    return total


def _require_pinned(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    # an empty tensor has no storage to pin and is never read
    if t.device.type != "cpu" or (t.numel() > 0 and not t.is_pinned()):
        raise ValueError(f"{name} must be a pinned (page-locked) CPU tensor")
    if t.dtype not in _U32_DTYPES:
        raise TypeError(f"{name} must have dtype in {_U32_DTYPES}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _scan_host(name: str, host_in: torch.Tensor, host_out, total, device, stream, workspace):
    _require_pinned(host_in, "host_in")
    if host_out is None:
        host_out = torch.empty_like(host_in).pin_memory()
    _require_pinned(host_out, "host_out")
    if host_out.numel() != host_in.numel():
        raise ValueError("host_in and host_out differ in length")
    if total is None:
        total = torch.empty(1, dtype=host_in.dtype).pin_memory()
    _require_pinned(total, "total")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    n = host_in.numel()
    with torch.cuda.device(device):
        sh = _stream_handle(stream)
        ws = _ws(_native.OP_SCAN_HOST, n, device, sh, workspace)
        fn = getattr(_native.lib(), name)
        _native.check(fn(host_in.data_ptr(), host_out.data_ptr(), n, total.data_ptr(), ws.ptr, ws.nbytes, sh), name)
    return host_out, total


def scan_exclusive_u32_host(host_in: torch.Tensor, host_out: torch.Tensor | None = None,
                            total: torch.Tensor | None = None, *, device=None, stream=None,
                            workspace: Workspace | None = None):
    """Exclusive scan of a pinned host array into a pinned host array (may be
    host_in itself), through the device. Asynchronous on the stream: the
    outputs are complete once the stream reaches the call. Returns
    (host_out, total), total a one-element pinned tensor."""
    return _scan_host("scan_exclusive_u32_host", host_in, host_out, total, device, stream, workspace)


def scan_inclusive_u32_host(host_in: torch.Tensor, host_out: torch.Tensor | None = None,
                            total: torch.Tensor | None = None, *, device=None, stream=None,
                            workspace: Workspace | None = None):
    """Inclusive scan of a pinned host array; otherwise as
    scan_exclusive_u32_host."""
    return _scan_host("scan_inclusive_u32_host", host_in, host_out, total, device, stream, workspace)


def scan_u32_op(data: torch.Tensor, op: str, inclusive: bool = False, total: torch.Tensor | None = None, *,
                stream=None, workspace: Workspace | None = None) -> torch.Tensor:
    """In place scan under op in {add, mul, and, or, xor, min, max} (u32;
    add and mul wrap). Returns the one-element device tensor holding the
    fold of all elements."""
    if op not in _native.SCAN_OPS:
        raise ValueError(f"op must be one of {sorted(_native.SCAN_OPS)}")
    _require_cuda(data, "data")
    total = _scalar_out(total, data, data.dtype)
    n = data.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_SCAN, n, data.device, sh, workspace)
    _native.check(_native.lib().scan_u32_op(_native.SCAN_OPS[op], int(bool(inclusive)), data.data_ptr(), n,
                                            total.data_ptr(), ws.ptr, ws.nbytes, sh), "scan_u32_op")
    return total


def scan_u64_op(data: torch.Tensor, op: str = "add", inclusive: bool = False, total: torch.Tensor | None = None,
                *, stream=None, workspace: Workspace | None = None) -> torch.Tensor:
    """In place scan of a 64-bit row (int64 or uint64 bits) under op in
    {add, mul, and, or, xor, min, max}, unsigned, add and mul wrapping at
    2^64. Returns the one-element device tensor holding the fold."""
    if op not in _native.SCAN_OPS:
        raise ValueError(f"op must be one of {sorted(_native.SCAN_OPS)}")
    u64 = (torch.int64, getattr(torch, "uint64", torch.int64))
    _require_cuda(data, "data", u64)
    if total is None:
        total = torch.empty(1, dtype=data.dtype, device=data.device)
    _require_cuda(total, "total", u64)
    n = data.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_SCAN64, n, data.device, sh, workspace)
    _native.check(_native.lib().scan_u64_op(_native.SCAN_OPS[op], int(bool(inclusive)), data.data_ptr(), n,
                                            total.data_ptr(), ws.ptr, ws.nbytes, sh), "scan_u64_op")
    return total


def _seg_args(data, head_flags, seg_sums, nseg):
    _require_cuda(data, "data")
    _require_cuda(head_flags, "head_flags", (torch.int32, torch.uint8))
    if head_flags.numel() != data.numel():
        raise ValueError("data and head_flags differ in length")
    if seg_sums is not None:
        _require_cuda(seg_sums, "seg_sums")
    nseg = _scalar_out(nseg, data, data.dtype)
    return nseg


def segscan_inclusive_u32(data: torch.Tensor, head_flags: torch.Tensor, seg_sums: torch.Tensor | None = None,
                          nseg: torch.Tensor | None = None, *, stream=None,
                          workspace: Workspace | None = None) -> torch.Tensor:
    """In place: data[j] <- sum of data over j's segment up to j (mod 2^32);
    a non-zero head flag (int32 or uint8) opens a segment, index 0 always does. If seg_sums
    is given, seg_sums[k] <- segment k's sum (for k < seg_sums.numel()).
    Returns the one-element device tensor holding the segment count."""
    nseg = _seg_args(data, head_flags, seg_sums, nseg)
    n = data.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_SEGSCAN, n, data.device, sh, workspace)
    name = "segscan_inclusive_u32" + ("_u8heads" if head_flags.dtype == torch.uint8 else "")
    _native.check(getattr(_native.lib(), name)(
        data.data_ptr(), head_flags.data_ptr(), n, seg_sums.data_ptr() if seg_sums is not None else None,
        seg_sums.numel() if seg_sums is not None else 0, nseg.data_ptr(), ws.ptr, ws.nbytes, sh), name)
    return nseg


def segreduce_u32(data: torch.Tensor, head_flags: torch.Tensor, seg_sums: torch.Tensor | None = None,
                  nseg: torch.Tensor | None = None, *, stream=None, workspace: Workspace | None = None):
    """Per-segment wrapped sums without writing the scan. seg_sums defaults
    to a fresh tensor of n elements (enough for any flag pattern). Returns
    (seg_sums, nseg): the first nseg entries of seg_sums are the sums."""
    if seg_sums is None:
        _require_cuda(data, "data")
        seg_sums = torch.empty(max(data.numel(), 1), dtype=data.dtype, device=data.device)
    nseg = _seg_args(data, head_flags, seg_sums, nseg)
    n = data.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_SEGSCAN, n, data.device, sh, workspace)
    name = "segreduce_u32" + ("_u8heads" if head_flags.dtype == torch.uint8 else "")
    _native.check(getattr(_native.lib(), name)(
        data.data_ptr(), head_flags.data_ptr(), n, seg_sums.data_ptr(), seg_sums.numel(), nseg.data_ptr(),
        ws.ptr, ws.nbytes, sh), name)
    return seg_sums, nseg


def compact_indices_u32(flags: torch.Tensor, offsets: torch.Tensor | None = None,
                        indices: torch.Tensor | None = None, count: torch.Tensor | None = None, *,
                        want_offsets: bool = True, stream=None, workspace: Workspace | None = None):
    """Stream compaction of int32 flags (non-zero keeps an element).
    Returns (offsets, indices, count): inclusive offsets (None when
    want_offsets is False and none were given), the kept indices at the
    front of `indices` with -1 after them, and the one-element count."""
    _require_cuda(flags, "flags", (torch.int32,))
    n = flags.numel()
    if offsets is None and want_offsets:
        offsets = torch.empty(n, dtype=torch.int32, device=flags.device)
    if offsets is not None:
        _require_cuda(offsets, "offsets", (torch.int32,))
        if offsets.numel() != n:
            raise ValueError("offsets must have n elements")
    if indices is None:
        indices = torch.empty(n, dtype=torch.int32, device=flags.device)
    _require_cuda(indices, "indices", (torch.int32,))
    if indices.numel() != n:
        raise ValueError("indices must have n elements")
    count = _scalar_out(count, flags, torch.int32)
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_COMPACT, n, flags.device, sh, workspace)
    _native.check(_native.lib().compact_indices_u32(
        flags.data_ptr(), n, offsets.data_ptr() if offsets is not None else None, indices.data_ptr(),
        count.data_ptr(), ws.ptr, ws.nbytes, sh), "compact_indices_u32")
    return offsets, indices, count


def compact_indices_u32_carry(flags: torch.Tensor, kept_before: torch.Tensor | None,
                              first_index: torch.Tensor | None, offsets: torch.Tensor | None = None,
                              indices: torch.Tensor | None = None, count: torch.Tensor | None = None, *,
                              stream=None, workspace: Workspace | None = None):
    """compact_indices_u32 of one piece of a longer flag array: kept_before
    and first_index (one-element int32 device tensors, or None for 0) are
    the kept elements and the elements before the piece. Returns (offsets,
    indices, count) as compact_indices_u32, with whole-array offsets and
    indices and the piece's own count."""
    _require_cuda(flags, "flags", (torch.int32,))
    for name, t in (("kept_before", kept_before), ("first_index", first_index)):
        if t is not None:
            _require_cuda(t, name, (torch.int32,))
            if t.numel() < 1:
                raise ValueError(f"{name} must hold at least one element")
    n = flags.numel()
    if offsets is None:
        offsets = torch.empty(n, dtype=torch.int32, device=flags.device)
    _require_cuda(offsets, "offsets", (torch.int32,))
    if indices is None:
        indices = torch.empty(n, dtype=torch.int32, device=flags.device)
    _require_cuda(indices, "indices", (torch.int32,))
    if offsets.numel() != n or indices.numel() != n:
        raise ValueError("offsets and indices must have n elements")
    count = _scalar_out(count, flags, torch.int32)
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_COMPACT, n, flags.device, sh, workspace)
    _native.check(_native.lib().compact_indices_u32_carry(
        flags.data_ptr(), n, kept_before.data_ptr() if kept_before is not None else None,
        first_index.data_ptr() if first_index is not None else None, offsets.data_ptr(), indices.data_ptr(),
        count.data_ptr(), ws.ptr, ws.nbytes, sh), "compact_indices_u32_carry")
    return offsets, indices, count


def segscan_piece_summary_u32(scanned: torch.Tensor, head_flags: torch.Tensor, nseg: torch.Tensor,
                              first_opens: bool, summary: torch.Tensor | None = None, *,
                              stream=None) -> torch.Tensor:
    """A piece's summary after segscan_inclusive_u32: (has head, tail,
    segments starting in it), three words in a device tensor."""
    _require_cuda(scanned, "scanned")
    _require_cuda(head_flags, "head_flags", (torch.int32,))
    _require_cuda(nseg, "nseg")
    if head_flags.numel() != scanned.numel():
        raise ValueError("head_flags must have as many elements as scanned")
    if summary is None:
        summary = torch.empty(3, dtype=torch.int32, device=scanned.device)
    _require_cuda(summary, "summary")
    if summary.numel() < 3:
        raise ValueError("summary must hold three elements")
    _native.check(_native.lib().segscan_piece_summary_u32(
        scanned.data_ptr(), head_flags.data_ptr(), scanned.numel(), nseg.data_ptr(), int(bool(first_opens)),
        summary.data_ptr(), _stream_handle(stream)), "segscan_piece_summary_u32")
    return summary


def segscan_piece_carries_u32(summaries: torch.Tensor, carries: torch.Tensor | None = None,
                              nseg_total: torch.Tensor | None = None, *, stream=None):
    """From g pieces' summaries (3 g words, in piece order): each piece's
    carry-in and the whole array's segment count (device tensors)."""
    _require_cuda(summaries, "summaries")
    if summaries.numel() % 3:
        raise ValueError("summaries must hold three words a piece")
    g = summaries.numel() // 3
    if carries is None:
        carries = torch.empty(g, dtype=torch.int32, device=summaries.device)
    _require_cuda(carries, "carries")
    nseg_total = _scalar_out(nseg_total, summaries, torch.int32)
    _native.check(_native.lib().segscan_piece_carries_u32(summaries.data_ptr(), g, carries.data_ptr(),
                                                          nseg_total.data_ptr(), _stream_handle(stream)),
                  "segscan_piece_carries_u32")
    return carries, nseg_total


def segscan_fix_u32(data: torch.Tensor, head_flags: torch.Tensor, carry: torch.Tensor, *, stream=None,
                    workspace: Workspace | None = None) -> torch.Tensor:
    """Adds carry (one-element device tensor) to the elements of the scanned
    piece before its first head. Returns data."""
    _require_cuda(data, "data")
    _require_cuda(head_flags, "head_flags", (torch.int32,))
    _require_cuda(carry, "carry")
    if head_flags.numel() != data.numel():
        raise ValueError("head_flags must have as many elements as data")
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_REDUCE, data.numel(), data.device, sh, workspace)
    _native.check(_native.lib().segscan_fix_u32(data.data_ptr(), head_flags.data_ptr(), data.numel(),
                                                carry.data_ptr(), ws.ptr, ws.nbytes, sh), "segscan_fix_u32")
    return data


def count_nonzero_u32(data: torch.Tensor, count: torch.Tensor | None = None, *, stream=None,
                      workspace: Workspace | None = None) -> torch.Tensor:
    """The number of non-zero elements of data (u32 or int32 flags), read
    once. Returns a one-element device tensor."""
    _require_cuda(data, "data")
    count = _scalar_out(count, data, data.dtype)
    n = data.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_REDUCE, n, data.device, sh, workspace)
    _native.check(_native.lib().count_nonzero_u32(data.data_ptr(), n, count.data_ptr(), ws.ptr, ws.nbytes, sh),
                  "count_nonzero_u32")
    return count


def fill_splitmix_u32(n: int, seed: int, stream_id: int = 0, start: int = 0, *, device=None,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The seeded input u32(seed, stream_id, start + i), i < n, drawn on the
    device: the same numbers as inputs.splitmix_u32 (counter-based
    SplitMix64), without a copy from the host. Returns an int32 tensor
    holding the u32 bits (out, when given, is filled and returned)."""
    if out is None:
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        out = torch.empty(n, dtype=torch.int32, device=dev)
    _require_cuda(out, "out")
    if out.numel() != n:
        raise ValueError("out must hold n elements")
    sh = _stream_handle(stream)
    _native.check(_native.lib().u32scan_fill_splitmix_u32(out.data_ptr(), n, seed, stream_id, start, sh),
                  "u32scan_fill_splitmix_u32")
    return out


def compact_values_u32(values: torch.Tensor, flags: torch.Tensor | None = None, out: torch.Tensor | None = None,
                       count: torch.Tensor | None = None, *, stream=None, workspace: Workspace | None = None):
    """The kept values, in order, at the front of `out` (the rest of out is
    left as it was); an element is kept when its flag is non-zero, or, with
    no flags, when its value is. Returns (out, count)."""
    _require_cuda(values, "values")
    n = values.numel()
    if flags is not None:
        _require_cuda(flags, "flags", (torch.int32,))
        if flags.numel() != n:
            raise ValueError("values and flags differ in length")
    if out is None:
        out = torch.empty_like(values)
    _require_cuda(out, "out")
    if out.numel() != n:
        raise ValueError("out must have n elements")
    count = _scalar_out(count, values, torch.int32)
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_COMPACT, n, values.device, sh, workspace)
    _native.check(_native.lib().compact_values_u32(values.data_ptr(), flags.data_ptr() if flags is not None else None,
                                                   n, out.data_ptr(), count.data_ptr(), ws.ptr, ws.nbytes, sh),
                  "compact_values_u32")
    return out, count


def radix_sort_perm_u32(keys: torch.Tensor, perm: torch.Tensor | None = None, *, stream=None,
                        workspace: Workspace | None = None) -> torch.Tensor:
    """The stable sorting permutation of u32 keys (int32 or uint32 tensor,
    unsigned order): keys[perm] is non-decreasing, ties by index."""
    _require_cuda(keys, "keys")
    n = keys.numel()
    if perm is None:
        perm = torch.empty(n, dtype=torch.int32, device=keys.device)
    _require_cuda(perm, "perm", (torch.int32,))
    if perm.numel() != n:
        raise ValueError("perm must have n elements")
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_RADIX, n, keys.device, sh, workspace)
    _native.check(_native.lib().radix_sort_perm_u32(keys.data_ptr(), n, perm.data_ptr(), ws.ptr, ws.nbytes, sh),
                  "radix_sort_perm_u32")
    return perm


def radix_sort_u32(keys: torch.Tensor, keys_out: torch.Tensor | None = None, perm: torch.Tensor | None = None,
                   *, want_perm: bool = True, stream=None, workspace: Workspace | None = None):
    """Stable radix sort of u32 keys (unsigned order). Returns (keys_out,
    perm): the sorted keys and, unless want_perm is False and no perm was
    given, the stable permutation (keys_out = keys[perm])."""
    _require_cuda(keys, "keys")
    n = keys.numel()
    if keys_out is None:
        keys_out = torch.empty_like(keys)
    _require_cuda(keys_out, "keys_out")
    if keys_out.numel() != n:
        raise ValueError("keys_out must have n elements")
    if perm is None and want_perm:
        perm = torch.empty(n, dtype=torch.int32, device=keys.device)
    if perm is not None:
        _require_cuda(perm, "perm", (torch.int32,))
        if perm.numel() != n:
            raise ValueError("perm must have n elements")
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_RADIX, n, keys.device, sh, workspace)
    _native.check(_native.lib().radix_sort_u32(keys.data_ptr(), n, keys_out.data_ptr(),
                                               perm.data_ptr() if perm is not None else None, ws.ptr, ws.nbytes, sh),
                  "radix_sort_u32")
    return keys_out, perm


def runs_layout_u32(counts: torch.Tensor, entries: torch.Tensor | None = None, slots: torch.Tensor | None = None,
                    *, stream=None, workspace: Workspace | None = None) -> torch.Tensor:
    """In place: counts[i] <- ends[i] = counts[0] + .. + counts[i] (mod
    2^32). Returns the one-element device tensor entries = max(total, 1);
    when given, slots[0 : min(entries, slots.numel())] is set to -1."""
    _require_cuda(counts, "counts")
    entries = _scalar_out(entries, counts, counts.dtype)
    if slots is not None:
        _require_cuda(slots, "slots", (torch.int32,))
    n = counts.numel()
    sh = _stream_handle(stream)
    ws = _ws(_native.OP_RUNS, n, counts.device, sh, workspace)
    _native.check(_native.lib().runs_layout_u32(counts.data_ptr(), n, entries.data_ptr(),
                                                slots.data_ptr() if slots is not None else None,
                                                slots.numel() if slots is not None else 0, ws.ptr, ws.nbytes, sh),
                  "runs_layout_u32")
    return entries


def runs_owner_u32(ends: torch.Tensor, owner: torch.Tensor | None = None, capacity: int | None = None, *,
                   stream=None) -> torch.Tensor:
    """owner[e] = the owner whose run holds entry e (the least i with
    e < ends[i]) for e in [0, min(entries, capacity)); -1 for the one slot of
    an empty layout. With no `owner` tensor, one of `capacity` elements is
    made (capacity defaults to entries, read back from the device)."""
    _require_cuda(ends, "ends")
    n = ends.numel()
    if owner is None:
        if capacity is None:
            total = int(ends[-1].item()) & 0xFFFFFFFF if n else 0
            capacity = max(total, 1)
        owner = torch.empty(capacity, dtype=torch.int32, device=ends.device)
    _require_cuda(owner, "owner", (torch.int32,))
    cap = owner.numel() if capacity is None else min(int(capacity), owner.numel())
    sh = _stream_handle(stream)
    _native.check(_native.lib().runs_owner_u32(ends.data_ptr(), n, owner.data_ptr(), cap, sh), "runs_owner_u32")
    return owner


def check(stream=None, workspace: Workspace | None = None, device=None) -> int:
    """Synchronise the stream and raise if a kernel that used the stream's
    cached workspace reported a device-side error (a carry-wait timeout)."""
    sh = _stream_handle(stream)
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        workspace = Workspace._cache.get((dev.index, sh))
        if workspace is None:
            torch.cuda.synchronize()
            return _native.OK
    status = _native.lib().u32scan_check(workspace.ptr, sh)
    _native.check(status, "u32scan_check")
    return status

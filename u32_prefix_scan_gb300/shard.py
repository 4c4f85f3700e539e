"""Scans of one U32 array split across ranks, one contiguous shard a rank.

Source: "scan.bend source", header comment (pass 2 scans the block sums) and
section Driver: the blocks are summed, the block sums are scanned, and each
block is rescanned from its base. Here the blocks are the ranks' shards, in
rank order (rank r holds the r-th piece of the array; pieces may differ in
length, and may be empty):

  1. every rank folds its shard to its wrapped sum (reduce_u32_op: 4 bytes
     read an element);
  2. one all-gather of the G shard sums (G words: all that crosses between
     GPUs);
  3. the exclusive scan of the gathered row (scan_exclusive_u32, on the
     device) gives rank r its carry-in, the wrapped sum of every element on
     the ranks before it, and the row's total is the whole array's;
  4. every rank scans its shard from its carry-in (scan_*_u32_carry: 8 bytes
     an element).

So a sharded scan moves 12 bytes an element against 8 on one GPU, with one
collective of G words and no host round trip. Sums wrap at 2^32 and are
associative, so the result has the bits of a one-GPU scan of the whole
array.

The compaction of a sharded flag array (the entelechy `compact` graph)
composes the same way: every rank counts its kept flags (count_nonzero_u32,
4 bytes read an element), one all-gather collects the G (count, length)
pairs, their exclusive scans give rank r the kept elements and the elements
before its shard, and every rank compacts its shard from those two device
words (compact_indices_u32_carry: whole-array offsets and kept indices, 12
bytes an element). The whole array's compacted indices are the ranks'
kept fronts in rank order.

The segmented scan of a sharded array ("Futhark.Pass.ExtractKernels.
Segmented", regularSegmentedScan) scans first and fixes after: every rank
scans its shard on its own (segscan_inclusive_u32, 12 bytes an element),
sums it up as (holds a head, scanned value at its end, segments starting in
it), one all-gather collects the G summaries, their segmented exclusive
scan gives each rank its carry-in, and the fix adds the carry-in to the
shard's elements before its first head (usually a short run; all of the
shard when it holds no head).

The composition takes its three local steps from a `steps` object (fold a
shard, scan the gathered row in place, scan a shard from a carry-in): by
default this library's kernels on CUDA tensors; the CPU tests pass other
implementations of the same steps and run the composition on gloo ranks.
This module only sequences the steps and the collective; it does no
arithmetic on the data itself.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


class KernelSteps:
    """The three local steps as this library's kernels (CUDA tensors)."""

    def __init__(self, workspace: api.Workspace | None = None):
        self.workspace = workspace

    def reduce(self, shard: torch.Tensor) -> torch.Tensor:
        return api.reduce_u32_op(shard, "add", workspace=self.workspace)

    def scan_row(self, row: torch.Tensor) -> torch.Tensor:
        return api.scan_exclusive_u32(row, workspace=self.workspace)

    def scan_from(self, shard: torch.Tensor, carry: torch.Tensor, inclusive: bool) -> torch.Tensor:
        fn = api.scan_inclusive_u32_carry if inclusive else api.scan_exclusive_u32_carry
        return fn(shard, carry, workspace=self.workspace)

    def segscan(self, shard: torch.Tensor, flags: torch.Tensor) -> torch.Tensor:
        return api.segscan_inclusive_u32(shard, flags, workspace=self.workspace)

    def summary(self, shard: torch.Tensor, flags: torch.Tensor, nseg: torch.Tensor, first: bool) -> torch.Tensor:
        return api.segscan_piece_summary_u32(shard, flags, nseg, first)

    def carries(self, summaries: torch.Tensor):
        return api.segscan_piece_carries_u32(summaries)

    def fix(self, shard: torch.Tensor, flags: torch.Tensor, carry: torch.Tensor) -> None:
        api.segscan_fix_u32(shard, flags, carry, workspace=self.workspace)

    def count(self, flags: torch.Tensor) -> torch.Tensor:
        return api.count_nonzero_u32(flags, workspace=self.workspace)

    def compact_from(self, flags: torch.Tensor, kept_before: torch.Tensor, first_index: torch.Tensor):
        return api.compact_indices_u32_carry(flags, kept_before, first_index, workspace=self.workspace)


def _all_gather(x: torch.Tensor, group) -> torch.Tensor:
    """The group's ranks' copies of the small 1-D tensor x, one after another
    in rank order, as one row."""
    world = dist.get_world_size(group)
    if dist.get_backend(group) == "nccl":
        row = torch.empty(world * x.numel(), dtype=x.dtype, device=x.device)
        dist.all_gather_into_tensor(row, x, group=group)
        return row
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x, group=group)
    return torch.cat(parts)


def sharded_scan(shard: torch.Tensor, inclusive: bool = False, group=None, steps=None, marks=None) -> torch.Tensor:
    """Scan this rank's shard in place as its piece of the whole array's
    exclusive (or inclusive) scan. Every rank of `group` calls it, in the
    same order as its other collectives. Returns the whole array's wrapped
    total (one-element tensor, on the shard's device), the same on every rank.
    `marks`: an optional pair of CUDA events recorded on the current stream
    just before and after the scan from the carry-in (for timing it).
    """
    steps = KernelSteps() if steps is None else steps
    rank = dist.get_rank(group)
    own = steps.reduce(shard)
    row = _all_gather(own.reshape(1), group)
    whole = steps.scan_row(row)  # row now holds each rank's carry-in
    if marks is not None:
        marks[0].record()
    steps.scan_from(shard, row[rank:rank + 1], inclusive)
    if marks is not None:
        marks[1].record()
    return whole


def sharded_compact(flags: torch.Tensor, group=None, steps=None, marks=None):
    """Compact this rank's shard of int32 flags as its piece of the whole
    array's compaction. Every rank of `group` calls it. Returns (offsets,
    indices, count, total): whole-array inclusive offsets for the shard, the
    shard's kept whole-array indices at the front of `indices` (-1 after
    them), the shard's kept count, and the whole array's kept count (the same
    on every rank). The whole array must hold fewer than 2^31 elements.
    `marks`: an optional pair of CUDA events recorded around the shard's
    compaction (for timing it)."""
    steps = KernelSteps() if steps is None else steps
    rank = dist.get_rank(group)
    own = steps.count(flags).reshape(1).to(torch.int32)
    length = torch.full((1,), flags.numel(), dtype=torch.int32, device=flags.device)
    row = _all_gather(torch.cat([own, length]), group)  # (count, length) of each rank, in rank order
    counts, lengths = row[0::2].contiguous(), row[1::2].contiguous()
    total = steps.scan_row(counts)  # counts now hold the kept elements before each rank
    steps.scan_row(lengths)  # lengths now hold each rank's first whole-array index
    if marks is not None:
        marks[0].record()
    offsets, indices, count = steps.compact_from(flags, counts[rank:rank + 1], lengths[rank:rank + 1])
    if marks is not None:
        marks[1].record()
    return offsets, indices, count, total


def sharded_segscan(shard: torch.Tensor, head_flags: torch.Tensor, group=None, steps=None,
                    marks=None) -> torch.Tensor:
    """Segmented inclusive scan of this rank's shard, in place, as its piece
    of the whole array's (a non-zero flag opens a segment; the whole array's
    element 0 opens one). Every rank of `group` calls it. Returns the whole
    array's segment count (one-element tensor), the same on every rank.
    `marks`: an optional pair of CUDA events recorded around the shard's own
    segmented scan (for timing it)."""
    steps = KernelSteps() if steps is None else steps
    rank = dist.get_rank(group)
    if marks is not None:
        marks[0].record()
    nseg = steps.segscan(shard, head_flags)
    if marks is not None:
        marks[1].record()
    own = steps.summary(shard, head_flags, nseg, rank == 0).reshape(3)
    row = _all_gather(own, group)  # the G summaries, in rank order
    carries, total = steps.carries(row)
    steps.fix(shard, head_flags, carries[rank:rank + 1])
    return total

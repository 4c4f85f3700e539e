"""The sharded scan's composition on two gloo ranks (CPU, no GPU).

u32_prefix_scan_gb300.shard.sharded_scan splits one array's scan across
ranks: each rank folds its shard, the shard sums are all-gathered, their
exclusive scan gives each rank its carry-in, and each rank scans its shard
from it ("scan.bend source", section Driver, one level up). Here the three
local steps are taken by the CPU oracle (fold = the oracle scan's total; a
scan from a carry-in = the oracle scan of the shard plus the carry) and the
exchange is a real gloo all-gather between two processes; the shards put
back together must equal the oracle's scan of the whole array, bit for bit.
"""

import json
import os
import socket

import numpy as np
import pytest

import oracle
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _u32(t):
    return t.numpy().view(np.uint32)


class OracleSteps:
    """The composition's local steps, computed by the CPU oracle."""

    def reduce(self, shard):
        return torch.from_numpy(np.array([oracle.scan_exclusive(_u32(shard))[1]], np.uint32).view(np.int32))

    def scan_row(self, row):
        out, total = oracle.scan_exclusive(_u32(row))
        row.copy_(torch.from_numpy(out.view(np.int32)))
        return torch.from_numpy(np.array([total], np.uint32).view(np.int32))

    def scan_from(self, shard, carry, inclusive):
        out, total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(_u32(shard))
        c = _u32(carry)[0]
        shard.copy_(torch.from_numpy((out + c).astype(np.uint32).view(np.int32)))  # wraps mod 2^32
        return torch.from_numpy(np.array([total + c], np.uint64).astype(np.uint32).view(np.int32))

    # the segmented scan's local steps, from their definitions
    def segscan(self, shard, flags):
        a, f = _u32(shard).copy(), flags.numpy()
        shard.copy_(torch.from_numpy(oracle.segscan_inclusive(a, f).view(np.int32)))
        return torch.tensor([oracle.segreduce(a, f)[1]], dtype=torch.int32)

    def summary(self, shard, flags, nseg, first):
        f = flags.numpy()
        if f.size == 0:
            return torch.zeros(3, dtype=torch.int32)
        local = int(nseg[0])
        has_head = int(local > 1 or f[0] != 0)
        return torch.tensor([has_head, int(_u32(shard)[-1]), local if (first or f[0] != 0) else local - 1],
                            dtype=torch.int64).to(torch.int32)

    def carries(self, row):
        r = _u32(row).reshape(-1, 3).astype(np.uint64)
        c, out = 0, []
        for has_head, tail, _ in r:
            out.append(c)
            c = int(tail) if has_head else (c + int(tail)) % (1 << 32)
        return (torch.from_numpy(np.array(out, np.uint32).view(np.int32)),
                torch.tensor([int(r[:, 2].sum())], dtype=torch.int32))

    def fix(self, shard, flags, carry):
        f = flags.numpy()
        first = int(np.flatnonzero(f)[0]) if np.any(f) else f.size
        a = _u32(shard).copy()
        a[:first] += _u32(carry)[0]  # wraps mod 2^32
        shard.copy_(torch.from_numpy(a.view(np.int32)))

    def count(self, flags):
        return torch.tensor([oracle.compact_indices(flags.numpy())[2]], dtype=torch.int32)

    def compact_from(self, flags, kept_before, first_index):
        # the shard's compaction as part of the whole array: offsets from the
        # kept elements before it, indices from the shard's first index
        off, idx, cnt = oracle.compact_indices(flags.numpy())
        kb, ib = int(kept_before[0]), int(first_index[0])
        idx = idx.copy()
        idx[:cnt] += ib
        return (torch.from_numpy((off + kb).astype(np.int32)), torch.from_numpy(idx.astype(np.int32)),
                torch.tensor([cnt], dtype=torch.int32))


CASES = {
    "uneven": (100003, [40000, 60003]),
    "empty_first": (5000, [0, 5000]),
    "empty_last": (70001, [70001, 0]),
    "tiny": (3, [1, 2]),
}


def _rank_main(rank, world, port, out_dir, case, inclusive):
    import torch.distributed as dist

    from u32_prefix_scan_gb300 import shard as sh

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n, cuts = CASES[case]
        whole = inputs.splitmix_u32(77, 0, n)
        lo = sum(cuts[:rank])
        piece = torch.from_numpy(whole[lo:lo + cuts[rank]].view(np.int32).copy())
        total = sh.sharded_scan(piece, inclusive=inclusive, steps=OracleSteps())
        np.save(os.path.join(out_dir, f"rank{rank}.npy"), _u32(piece))
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
            json.dump({"total": int(_u32(total)[0])}, fh)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("inclusive", [False, True], ids=["exclusive", "inclusive"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_two_gloo_ranks_compose_the_whole_scan(tmp_path, case, inclusive):
    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_rank_main, args=(world, free_port(), str(tmp_path), case, inclusive), nprocs=world, join=True)
    n, _ = CASES[case]
    whole = inputs.splitmix_u32(77, 0, n)
    want, want_total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(whole)
    got = np.concatenate([np.load(tmp_path / f"rank{r}.npy") for r in range(world)])
    assert np.array_equal(got, want)
    for r in range(world):
        assert json.loads((tmp_path / f"rank{r}.json").read_text())["total"] == want_total


COMPACT_CASES = {
    "uneven": (100003, [40000, 60003], 0.1),
    "dense": (50001, [25000, 25001], 0.9),
    "empty_first": (7001, [0, 7001], 0.1),
}


def _compact_rank_main(rank, world, port, out_dir, case):
    import torch.distributed as dist

    from u32_prefix_scan_gb300 import shard as sh

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n, cuts, p = COMPACT_CASES[case]
        whole = inputs.compact_flags(n, 78, p)
        lo = sum(cuts[:rank])
        piece = torch.from_numpy(whole[lo:lo + cuts[rank]].copy())
        offsets, indices, count, total = sh.sharded_compact(piece, steps=OracleSteps())
        np.save(os.path.join(out_dir, f"off{rank}.npy"), offsets.numpy())
        np.save(os.path.join(out_dir, f"idx{rank}.npy"), indices.numpy()[:int(count[0])])
        np.save(os.path.join(out_dir, f"tail{rank}.npy"), indices.numpy()[int(count[0]):])
        with open(os.path.join(out_dir, f"c{rank}.json"), "w") as fh:
            json.dump({"total": int(total[0])}, fh)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(COMPACT_CASES))
def test_two_gloo_ranks_compose_the_whole_compaction(tmp_path, case):
    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_compact_rank_main, args=(world, free_port(), str(tmp_path), case), nprocs=world, join=True)
    n, _, p = COMPACT_CASES[case]
    want_off, want_idx, want_count = oracle.compact_indices(inputs.compact_flags(n, 78, p))
    got_off = np.concatenate([np.load(tmp_path / f"off{r}.npy") for r in range(world)])
    got_idx = np.concatenate([np.load(tmp_path / f"idx{r}.npy") for r in range(world)])
    assert np.array_equal(got_off, want_off)
    assert np.array_equal(got_idx, want_idx[:want_count])
    for r in range(world):
        assert (np.load(tmp_path / f"tail{r}.npy") == -1).all()
        assert json.loads((tmp_path / f"c{r}.json").read_text())["total"] == want_count


SEG_CASES = {
    "geometric": (100003, [40000, 60003], 6),
    "long_segments": (60001, [1000, 29000, 30001], 14),  # shards with no head at all
    "empty_middle": (7001, [3000, 0, 4001], 4),
}


def _seg_rank_main(rank, world, port, out_dir, case):
    import torch.distributed as dist

    from u32_prefix_scan_gb300 import shard as sh

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n, cuts, lg = SEG_CASES[case]
        a = inputs.splitmix_u32(79, 0, n)
        f = inputs.segment_heads_geometric(n, 79, log2_mean=lg)
        lo = sum(cuts[:rank])
        piece = torch.from_numpy(a[lo:lo + cuts[rank]].view(np.int32).copy())
        flags = torch.from_numpy(f[lo:lo + cuts[rank]].copy())
        total = sh.sharded_segscan(piece, flags, steps=OracleSteps())
        np.save(os.path.join(out_dir, f"s{rank}.npy"), _u32(piece))
        with open(os.path.join(out_dir, f"s{rank}.json"), "w") as fh:
            json.dump({"nseg": int(total[0])}, fh)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(SEG_CASES))
def test_gloo_ranks_compose_the_whole_segmented_scan(tmp_path, case):
    import torch.multiprocessing as mp

    n, cuts, lg = SEG_CASES[case]
    world = len(cuts)
    mp.spawn(_seg_rank_main, args=(world, free_port(), str(tmp_path), case), nprocs=world, join=True)
    a = inputs.splitmix_u32(79, 0, n)
    f = inputs.segment_heads_geometric(n, 79, log2_mean=lg)
    got = np.concatenate([np.load(tmp_path / f"s{r}.npy") for r in range(world)])
    assert np.array_equal(got, oracle.segscan_inclusive(a, f))
    for r in range(world):
        assert json.loads((tmp_path / f"s{r}.json").read_text())["nseg"] == oracle.segreduce(a, f)[1]

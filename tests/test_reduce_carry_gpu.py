"""GPU parity of the fold (reduce_u32_op), the scans from a carry-in
(scan_*_u32_carry) and their composition into a sharded scan, against the
CPU oracle, through the C ABI.

The fold is checked under every CAIRN integer operator against the oracle's
scan total; a scan from a carry-in c against the oracle scan plus c (the
scan of the piece as part of a longer array whose earlier elements sum to
c). The composition splits one array into pieces and scans each from the
exclusive scan of the pieces' folds ("scan.bend source", section Driver,
with pieces for blocks): the pieces put back together must equal the
oracle's scan of the whole array. On one GPU the pieces' exchange is
emulated by concatenation (no kernel waits on another), and the
collective-driven form runs on a one-rank NCCL group.
"""

import os
import socket

import numpy as np
import pytest

import oracle
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SIZES = [0, 1, 3, 4, 1000, 4 * 512 * 4 * 2 + 5, (1 << 20) + 3, (1 << 24) + 12345]


@pytest.fixture(scope="module")
def u():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import build

    build.build()
    import u32_prefix_scan_gb300 as u

    return u


def dev32(a, offset=0):
    buf = torch.empty(a.size + offset + 4, dtype=torch.int32, device="cuda")
    view = buf[offset: offset + a.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int32)))
    return view


def host_u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("op", ["add", "mul", "and", "or", "xor", "min", "max"])
@pytest.mark.parametrize("n", SIZES)
def test_fold_matches_the_oracle(u, op, n):
    a = inputs.splitmix_u32(61, 0, n)
    if op == "mul":
        a = a | 1  # odd factors: the product stays informative instead of reaching 0
    for offset in (0, 1, 3):  # every 4-byte phase of the start
        d = dev32(a, offset)
        total = u.reduce_u32_op(d, op)
        u.check()
        assert int(host_u32(total)[0]) == oracle.scan_op(a, op, False)[1], (op, n, offset)
        assert np.array_equal(host_u32(d), a)  # read only


@pytest.mark.parametrize("inclusive", [False, True], ids=["exclusive", "inclusive"])
@pytest.mark.parametrize("n", SIZES)
def test_scan_from_a_carry_in(u, n, inclusive):
    a = inputs.splitmix_u32(62, 0, n)
    c = np.uint32(0xDEADBEEF)
    want, want_total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(a)
    fn = u.scan_inclusive_u32_carry if inclusive else u.scan_exclusive_u32_carry
    for offset in (0, 2):
        d = dev32(a, offset)
        carry = torch.from_numpy(np.array([c], np.uint32).view(np.int32)).cuda()
        total = fn(d, carry)
        u.check()
        assert np.array_equal(host_u32(d), (want + c).astype(np.uint32)), (n, offset)
        assert int(host_u32(total)[0]) == (want_total + int(c)) % (1 << 32)
    # no carry-in: the plain scan
    d = dev32(a)
    total = fn(d, None)
    u.check()
    assert np.array_equal(host_u32(d), want) and int(host_u32(total)[0]) == want_total


@pytest.mark.parametrize("inclusive", [False, True], ids=["exclusive", "inclusive"])
@pytest.mark.parametrize("cuts", [[70001, 0, (1 << 22) + 9, 123], [(1 << 21) + 1, (1 << 21) + 1, 5]],
                         ids=["uneven-with-empty", "two-long-one-short"])
def test_pieces_scanned_from_their_carries_make_the_whole_scan(u, cuts, inclusive):
    from u32_prefix_scan_gb300.shard import KernelSteps

    whole = inputs.splitmix_u32(63, 0, sum(cuts))
    steps = KernelSteps()
    bounds = np.cumsum([0] + cuts)
    pieces = [dev32(whole[bounds[r]:bounds[r + 1]]) for r in range(len(cuts))]
    row = torch.cat([steps.reduce(p) for p in pieces])  # the all-gather, emulated
    grand = steps.scan_row(row)
    for r, p in enumerate(pieces):
        steps.scan_from(p, row[r:r + 1], inclusive)
    u.check()
    want, want_total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(whole)
    got = np.concatenate([host_u32(p) for p in pieces])
    assert np.array_equal(got, want)
    assert int(host_u32(grand)[0]) == want_total


def test_sharded_scan_on_a_one_rank_nccl_group(u):
    import torch.distributed as dist

    from u32_prefix_scan_gb300 import shard

    if dist.is_initialized():
        pytest.skip("a process group already exists")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        a = inputs.splitmix_u32(64, 0, (1 << 22) + 77)
        d = dev32(a)
        total = shard.sharded_scan(d)
        u.check()
        want, want_total = oracle.scan_exclusive(a)
        assert np.array_equal(host_u32(d), want) and int(host_u32(total)[0]) == want_total
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("p", [0.1, 0.9])
@pytest.mark.parametrize("n", [0, 1, 5, 1000, (1 << 20) + 3, (1 << 24) + 12345])
def test_count_nonzero_matches_the_oracle(u, n, p):
    f = inputs.compact_flags(n, 65, p)
    f[::7] = -7  # any non-zero flag keeps its element
    for offset in (0, 3):
        d = dev32(f.view(np.uint32), offset)
        count = u.count_nonzero_u32(d)
        u.check()
        assert int(host_u32(count)[0]) == oracle.compact_indices(f)[2], (n, offset)


@pytest.mark.parametrize("n", [1, 1000, 100003, (1 << 22) + 77])
def test_compaction_from_carry_ins(u, n):
    f = inputs.compact_flags(n, 66, 0.1)
    want_off, want_idx, want_cnt = oracle.compact_indices(f)
    kb = torch.tensor([12345], dtype=torch.int32, device="cuda")
    ib = torch.tensor([1 << 24], dtype=torch.int32, device="cuda")
    off, idx, cnt = u.compact_indices_u32_carry(dev32(f.view(np.uint32), 1).view(torch.int32), kb, ib)
    u.check()
    assert int(cnt.item()) == want_cnt
    assert np.array_equal(off.cpu().numpy(), want_off + 12345)
    got = idx.cpu().numpy()
    assert np.array_equal(got[:want_cnt], want_idx[:want_cnt] + (1 << 24)) and (got[want_cnt:] == -1).all()
    # no carry-ins: the plain compaction
    off, idx, cnt = u.compact_indices_u32_carry(dev32(f.view(np.uint32)).view(torch.int32), None, None)
    u.check()
    assert np.array_equal(off.cpu().numpy(), want_off) and np.array_equal(idx.cpu().numpy(), want_idx)


@pytest.mark.parametrize("cuts", [[70001, 0, (1 << 22) + 9, 123], [(1 << 21) + 1, (1 << 21) + 1, 5]],
                         ids=["uneven-with-empty", "two-long-one-short"])
def test_pieces_compacted_from_their_carries_make_the_whole_compaction(u, cuts):
    from u32_prefix_scan_gb300.shard import KernelSteps

    whole = inputs.compact_flags(sum(cuts), 67, 0.1)
    steps = KernelSteps()
    bounds = np.cumsum([0] + cuts)
    pieces = [dev32(whole[bounds[r]:bounds[r + 1]].view(np.uint32)).view(torch.int32) for r in range(len(cuts))]
    counts = torch.cat([steps.count(p) for p in pieces])  # the all-gather, emulated
    lengths = torch.tensor(cuts, dtype=torch.int32, device="cuda")
    grand = steps.scan_row(counts)
    steps.scan_row(lengths)
    got_off, got_idx = [], []
    for r, p in enumerate(pieces):
        off, idx, cnt = steps.compact_from(p, counts[r:r + 1], lengths[r:r + 1])
        k = int(cnt.item())
        got_off.append(off.cpu().numpy())
        got_idx.append(idx.cpu().numpy()[:k])
        assert (idx.cpu().numpy()[k:] == -1).all()
    u.check()
    want_off, want_idx, want_cnt = oracle.compact_indices(whole)
    assert np.array_equal(np.concatenate(got_off), want_off)
    assert np.array_equal(np.concatenate(got_idx), want_idx[:want_cnt])
    assert int(grand.item()) == want_cnt


def test_sharded_compaction_on_a_one_rank_nccl_group(u):
    import torch.distributed as dist

    from u32_prefix_scan_gb300 import shard

    if dist.is_initialized():
        pytest.skip("a process group already exists")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        f = inputs.compact_flags((1 << 22) + 77, 68, 0.9)
        off, idx, cnt, total = shard.sharded_compact(dev32(f.view(np.uint32)).view(torch.int32))
        u.check()
        want_off, want_idx, want_cnt = oracle.compact_indices(f)
        assert np.array_equal(off.cpu().numpy(), want_off) and np.array_equal(idx.cpu().numpy(), want_idx)
        assert int(cnt.item()) == want_cnt == int(total.item())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("lg", [6, 16], ids=["short-segments", "long-segments"])
@pytest.mark.parametrize("cuts", [[70001, 0, (1 << 22) + 9, 123], [(1 << 21) + 1, (1 << 21) + 1, 5]],
                         ids=["uneven-with-empty", "two-long-one-short"])
def test_pieces_segscanned_and_fixed_make_the_whole_segmented_scan(u, cuts, lg):
    """Pieces scanned on their own, summed up, their carries combined and
    the pieces fixed: the whole array's segmented scan and segment count
    (long segments leave whole pieces without a head)."""
    from u32_prefix_scan_gb300.shard import KernelSteps

    n = sum(cuts)
    a = inputs.splitmix_u32(69, 0, n)
    f = inputs.segment_heads_geometric(n, 69, log2_mean=lg)
    steps = KernelSteps()
    bounds = np.cumsum([0] + cuts)
    pieces = [dev32(a[bounds[r]:bounds[r + 1]]) for r in range(len(cuts))]
    flags = [dev32(f[bounds[r]:bounds[r + 1]].view(np.uint32)) for r in range(len(cuts))]
    summaries = []
    for r, (p, fl) in enumerate(zip(pieces, flags)):
        nseg = steps.segscan(p, fl)
        summaries.append(steps.summary(p, fl, nseg, r == 0))
    carries, total = steps.carries(torch.cat(summaries))  # the all-gather, emulated
    for r, (p, fl) in enumerate(zip(pieces, flags)):
        steps.fix(p, fl, carries[r:r + 1])
    u.check()
    got = np.concatenate([host_u32(p) for p in pieces])
    assert np.array_equal(got, oracle.segscan_inclusive(a, f))
    assert int(host_u32(total)[0]) == oracle.segreduce(a, f)[1]


@pytest.mark.parametrize("first_head", [0, 5, 8191, 8192, 100000, None])
def test_fix_adds_the_carry_before_the_first_head_only(u, first_head):
    n = (1 << 20) + 3
    a = inputs.splitmix_u32(70, 0, n)
    f = np.zeros(n, np.int32)
    if first_head is not None:
        f[first_head] = 1
        f[first_head + 1000::777] = -3
    d, fl = dev32(a), dev32(f.view(np.uint32))
    carry = torch.tensor([0x12345678], dtype=torch.int32, device="cuda")
    u.segscan_fix_u32(d, fl, carry)
    u.check()
    want = a.copy()
    stop = n if first_head is None else first_head
    want[:stop] += np.uint32(0x12345678)
    assert np.array_equal(host_u32(d), want)


def test_sharded_segscan_on_a_one_rank_nccl_group(u):
    import torch.distributed as dist

    from u32_prefix_scan_gb300 import shard

    if dist.is_initialized():
        pytest.skip("a process group already exists")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        n = (1 << 22) + 77
        a = inputs.splitmix_u32(71, 0, n)
        f = inputs.segment_heads_geometric(n, 71, log2_mean=10)
        d = dev32(a)
        total = shard.sharded_segscan(d, dev32(f.view(np.uint32)))
        u.check()
        assert np.array_equal(host_u32(d), oracle.segscan_inclusive(a, f))
        assert int(host_u32(total)[0]) == oracle.segreduce(a, f)[1]
    finally:
        dist.destroy_process_group()

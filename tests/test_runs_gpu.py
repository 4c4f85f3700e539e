"""GPU parity of the runs layout and of owner(e, ends) over every entry
against the CPU oracle, through the C ABI: uniform and skewed count mixes,
one long run, runs at the first and last owner only, no entries at all,
capacities below and above the entry count, sizes spanning many tiles with
ragged tails, and the benchmark workload at full size (n = 2^25 owners)."""

import numpy as np
import pytest

import oracle
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def u():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import build

    build.build()
    import u32_prefix_scan_gb300 as u

    return u


def counts_for(kind: str, n: int, seed: int = 6) -> np.ndarray:
    if kind == "uniform":
        return inputs.run_counts(n, seed)
    if kind == "skewed":
        return inputs.run_counts(n, seed, skewed=True)
    if kind == "zeros":
        return np.zeros(n, dtype=np.uint32)
    if kind == "ones":
        return np.ones(n, dtype=np.uint32)
    if kind == "one_long":  # a single owner in the middle holds every entry
        c = np.zeros(n, dtype=np.uint32)
        c[n // 2] = 300007
        return c
    if kind == "ends_only":  # only the first and the last owner hold entries
        c = np.zeros(n, dtype=np.uint32)
        c[0], c[-1] = 5000, 7
        return c
    if kind == "sparse_long":  # one owner in 4096 holds a run of up to 16383
        d = inputs.splitmix_u32(seed, 1, n)
        return np.where((d & np.uint32(4095)) == 0, d >> np.uint32(18), np.uint32(0)).astype(np.uint32)
    raise ValueError(kind)


def layout_and_owner(u, counts, slot_extra=3):
    ends_d = torch.from_numpy(counts.view(np.int32).copy()).cuda()
    want_ends, want_entries, want_owner = oracle.runs_owner(counts)
    slots = torch.full((want_entries + slot_extra,), 77, dtype=torch.int32, device="cuda")
    entries = u.runs_layout_u32(ends_d, slots=slots)
    u.check()
    assert np.array_equal(ends_d.cpu().numpy().view(np.uint32), want_ends)
    assert int(entries.item()) == want_entries
    s = slots.cpu().numpy()
    assert np.all(s[:want_entries] == -1) and np.all(s[want_entries:] == 77)
    return ends_d, want_entries, want_owner


SIZES = [1, 2, 31, 2047, 2048, 2049, 5000, 100003, (1 << 20) + 17]


@pytest.mark.parametrize("kind", ["uniform", "skewed", "ones", "one_long", "ends_only", "sparse_long"])
@pytest.mark.parametrize("n", SIZES)
def test_runs_layout_and_owner(u, kind, n):
    counts = counts_for(kind, n)
    ends_d, entries, want = layout_and_owner(u, counts)
    owner = torch.full((entries + 5,), 99, dtype=torch.int32, device="cuda")
    u.runs_owner_u32(ends_d, owner, capacity=entries + 5)
    torch.cuda.synchronize()
    got = owner.cpu().numpy()
    assert np.array_equal(got[:entries], want)
    assert np.all(got[entries:] == 99)  # nothing written past the entries


@pytest.mark.parametrize("n", [0, 1, 1000])
def test_runs_with_no_entries(u, n):
    counts = counts_for("zeros", n)
    ends_d, entries, want = layout_and_owner(u, counts)
    assert entries == 1 and want.tolist() == [-1]
    owner = torch.full((4,), 99, dtype=torch.int32, device="cuda")
    u.runs_owner_u32(ends_d, owner, capacity=4)
    torch.cuda.synchronize()
    assert owner.cpu().tolist() == [-1, 99, 99, 99]


@pytest.mark.parametrize("kind", ["uniform", "skewed", "one_long"])
@pytest.mark.parametrize("frac", [0.0, 0.001, 0.37, 0.999])
def test_owner_capacity_below_entries(u, kind, frac):
    counts = counts_for(kind, 100003)
    ends_d, entries, want = layout_and_owner(u, counts)
    cap = int(entries * frac)
    owner = torch.full((cap + 8,), 99, dtype=torch.int32, device="cuda")
    u.runs_owner_u32(ends_d, owner, capacity=cap)
    torch.cuda.synchronize()
    got = owner.cpu().numpy()
    assert np.array_equal(got[:cap], want[:cap]) and np.all(got[cap:] == 99)


def test_slots_capacity_below_entries(u):
    counts = counts_for("uniform", 50000)
    d = torch.from_numpy(counts.view(np.int32).copy()).cuda()
    slots = torch.full((1001,), 77, dtype=torch.int32, device="cuda")
    entries = u.runs_layout_u32(d, slots=slots[:1000])
    u.check()
    assert int(entries.item()) == int(counts.sum())
    s = slots.cpu().numpy()
    assert np.all(s[:1000] == -1) and s[1000] == 77


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_rows(u, offset):
    counts = counts_for("uniform", 70001)
    want_ends, entries, want = oracle.runs_owner(counts)
    buf = torch.zeros(counts.size + 4, dtype=torch.int32, device="cuda")
    d = buf[offset:offset + counts.size]
    d.copy_(torch.from_numpy(counts.view(np.int32)))
    sbuf = torch.full((entries + 8,), 77, dtype=torch.int32, device="cuda")
    e = u.runs_layout_u32(d, slots=sbuf[offset:offset + entries])
    obuf = torch.full((entries + 8,), 99, dtype=torch.int32, device="cuda")
    u.runs_owner_u32(d, obuf[offset:offset + entries])
    u.check()
    assert int(e.item()) == entries
    assert np.array_equal(d.cpu().numpy().view(np.uint32), want_ends)
    s = sbuf.cpu().numpy()
    assert np.all(s[offset:offset + entries] == -1) and np.all(s[:offset] == 77)
    o = obuf.cpu().numpy()
    assert np.array_equal(o[offset:offset + entries], want) and np.all(o[:offset] == 99)


def test_repeated_calls_share_one_workspace(u):
    ws = u.Workspace(1 << 20, torch.device("cuda"))
    for seed in range(4):
        counts = inputs.run_counts(300007, seed)
        d = torch.from_numpy(counts.view(np.int32).copy()).cuda()
        e = u.runs_layout_u32(d, workspace=ws)
        owner = u.runs_owner_u32(d)
        u.check()
        want_ends, entries, want = oracle.runs_owner(counts)
        assert int(e.item()) == entries
        assert np.array_equal(owner.cpu().numpy(), want)


@pytest.mark.parametrize("skewed", [False, True])
def test_full_size(u, skewed):
    counts = inputs.run_counts(1 << 25, 6, skewed=skewed)
    ends_d, entries, want = layout_and_owner(u, counts, slot_extra=0)
    owner = u.runs_owner_u32(ends_d)
    torch.cuda.synchronize()
    assert np.array_equal(owner.cpu().numpy(), want)

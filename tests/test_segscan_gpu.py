"""GPU parity of the segmented scan and per-segment reduce against the CPU
oracle, through the C ABI: bit-exact scans, sums and counts over head
patterns from one segment to all heads, geometric and length-4 segments,
ragged tails, misaligned and differently aligned streams, a capacity below
the segment count, repeated calls on one workspace, both benchmark
workloads at full size (n = 2^26), and the bounded carry wait (a tile that
never publishes its carry words is reported, and the workspace recovers)."""

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


def dev(a: np.ndarray, offset: int = 0):
    buf = torch.empty(a.size + offset + 4, dtype=torch.int32, device="cuda")
    view = buf[offset: offset + a.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int32)))
    return view


def host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def heads(kind: str, n: int, seed: int = 3) -> np.ndarray:
    if kind == "geometric":
        return inputs.segment_heads_geometric(n, seed)
    if kind == "geometric16":
        return inputs.segment_heads_geometric(n, seed, log2_mean=4)
    if kind == "regular4":
        return inputs.segment_heads_regular(n, 4)
    if kind == "regular7":
        return inputs.segment_heads_regular(n, 7)
    if kind == "all":
        return np.ones(n, np.int32)
    if kind == "none":
        return np.zeros(n, np.int32)
    if kind == "half":
        f = (inputs.splitmix_u32(seed, 1, n) < np.uint32(1 << 31)).astype(np.int32)
        f[f != 0] = np.where(np.arange(int(f.sum())) % 3 == 0, -5, 9)  # any non-zero value is a head
        return f
    raise ValueError(kind)


def check_segscan(u, a, f, offset_a=0, offset_f=0, cap=None):
    n = a.size
    d, fl = dev(a, offset_a), dev(f, offset_f)
    want_sums, want_nseg = oracle.segreduce(a, f)
    cap = max(n, 1) if cap is None else cap
    sums = torch.full((max(cap, 1),), -1, dtype=torch.int32, device="cuda")
    nseg = u.segscan_inclusive_u32(d, fl, sums[:cap] if cap else None)
    u.check()
    assert np.array_equal(host(d), oracle.segscan_inclusive(a, f))
    assert int(host(nseg)[0]) == want_nseg
    k = min(cap, want_nseg)
    assert np.array_equal(host(sums)[:k], want_sums[:k])
    assert np.all(host(sums)[k:cap] == 0xFFFFFFFF)  # nothing written past the segments / capacity
    # the form without sums (its own count path) on the same input
    d2 = dev(a, offset_a)
    c2 = u.segscan_inclusive_u32(d2, fl)
    u.check()
    assert np.array_equal(host(d2), host(d)) and int(host(c2)[0]) == want_nseg


# around the tiles of the forms that write the scan (10240 elements with
# int32 flags) and of the reduce (14336), with ragged tails
SIZES = [1, 2, 5, 4096 + 3, 10240, 10240 + 1, 3 * 10240 + 77, 14336 + 1, 3 * 14336 + 77, 100003, (1 << 20) + 5]


@pytest.mark.parametrize("kind", ["geometric", "geometric16", "regular4", "regular7", "all", "none", "half"])
@pytest.mark.parametrize("n", SIZES)
def test_segscan_parity(u, kind, n):
    check_segscan(u, inputs.scan_values(n, 3), heads(kind, n))


@pytest.mark.parametrize("offsets", [(1, 1), (2, 2), (3, 3), (1, 2), (0, 3), (3, 0)])
@pytest.mark.parametrize("n", [7, 10240 * 3 + 5, 14336 * 3 + 5, (1 << 18) + 3])
def test_segscan_misaligned(u, offsets, n):
    check_segscan(u, inputs.scan_values(n, 5), heads("half", n, 5), *offsets)


def test_segscan_capacity_below_count(u):
    n = 100003
    check_segscan(u, inputs.scan_values(n, 3), heads("geometric16", n), cap=1000)


@pytest.mark.parametrize("kind", ["geometric", "regular4", "half", "none"])
@pytest.mark.parametrize("n", [1, 14336 + 1, 3 * 14336 + 77, 100003, (1 << 20) + 5])
def test_segreduce_parity(u, kind, n):
    a, f = inputs.scan_values(n, 3), heads(kind, n)
    d, fl = dev(a), dev(f)
    sums, nseg = u.segreduce_u32(d, fl)
    u.check()
    want_sums, want_nseg = oracle.segreduce(a, f)
    assert int(host(nseg)[0]) == want_nseg
    assert np.array_equal(host(sums)[:want_nseg], want_sums)
    assert np.array_equal(host(d), a)  # the reduce leaves data as it was


@pytest.mark.parametrize("kind", ["regular4", "regular7", "half", "geometric16"])
@pytest.mark.parametrize("word_offset", [0, 1])
@pytest.mark.parametrize("cut", [False, True])
def test_segreduce_sums_at_any_word_and_capacity(u, kind, word_offset, cut):
    """The reduce writes a lane's consecutive segment sums two to a store
    where the index allows: sums rows at an even and an odd word (8-byte
    alignment or not), with the capacity at the count or cut to an odd
    number inside a lane's run of ends; nothing before the row or past the
    capacity is written."""
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    n = 3 * 14336 + 77
    a, f = inputs.scan_values(n, 9), heads(kind, n, 9)
    want_sums, want_nseg = oracle.segreduce(a, f)
    cap = (want_nseg // 2) | 1 if cut else want_nseg
    buf = torch.full((cap + word_offset + 4,), -1, dtype=torch.int32, device="cuda")
    sums = buf[word_offset: word_offset + cap]
    d, fl = dev(a), dev(f)
    nseg = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = u.Workspace(lib.u32scan_workspace_bytes(_native.OP_SEGSCAN, n), torch.device("cuda"))
    st = torch.cuda.current_stream().cuda_stream
    assert lib.segreduce_u32(d.data_ptr(), fl.data_ptr(), n, sums.data_ptr(), cap, nseg.data_ptr(), ws.ptr,
                             ws.nbytes, st) == _native.OK
    assert lib.u32scan_check(ws.ptr, st) == _native.OK
    assert int(nseg.item()) == want_nseg
    got = host(buf)
    assert np.array_equal(got[word_offset: word_offset + cap], want_sums[:cap])
    assert np.all(got[:word_offset] == 0xFFFFFFFF) and np.all(got[word_offset + cap:] == 0xFFFFFFFF)


def test_segreduce_count_only_and_empty(u):
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    n = 50000
    a, f = inputs.scan_values(n, 3), heads("geometric16", n)
    d, fl = dev(a), dev(f)
    nseg = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = u.Workspace(lib.u32scan_workspace_bytes(_native.OP_SEGSCAN, n), torch.device("cuda"))
    s = torch.cuda.current_stream().cuda_stream
    assert lib.segreduce_u32(d.data_ptr(), fl.data_ptr(), n, None, 0, nseg.data_ptr(), ws.ptr, ws.nbytes,
                             s) == _native.OK
    assert lib.u32scan_check(ws.ptr, s) == _native.OK
    assert int(nseg.item()) == oracle.segreduce(a, f)[1]
    nseg.fill_(7)
    assert lib.segscan_inclusive_u32(d.data_ptr(), fl.data_ptr(), 0, None, 0, nseg.data_ptr(), ws.ptr,
                                     ws.nbytes, s) == _native.OK
    torch.cuda.synchronize()
    assert int(nseg.item()) == 0


def test_repeated_calls_share_one_workspace(u):
    ws = u.Workspace(1 << 20, torch.device("cuda"))
    rng = np.random.default_rng(4)
    for k in range(24):
        n = int(rng.choice([1, 777, 8192 * 3, 100003, (1 << 20) + 5]))
        a = inputs.splitmix_u32(9, 0, n, start=k * 1000)
        f = heads(["geometric16", "regular4", "half"][k % 3], n, 9 + k)
        d, fl = dev(a), dev(f)
        if k % 2:
            sums, nseg = u.segreduce_u32(d, fl, workspace=ws)
            u.check(workspace=ws)
            want, cnt = oracle.segreduce(a, f)
            assert int(host(nseg)[0]) == cnt and np.array_equal(host(sums)[:cnt], want), k
        else:
            u.segscan_inclusive_u32(d, fl, workspace=ws)
            u.check(workspace=ws)
            assert np.array_equal(host(d), oracle.segscan_inclusive(a, f)), k


@pytest.mark.parametrize("kind", ["geometric", "regular4"])
def test_workload_2_26_full_parity(u, kind):
    # The segmented benchmark configurations: n = 2^26, values u32(3, 0, i),
    # heads Bernoulli(2^-10) (mean length 1024) or every 4th index.
    n = 1 << 26
    a = inputs.scan_values(n, 3)
    f = heads(kind, n)
    check_segscan(u, a, f)
    d, fl = dev(a), dev(f)
    sums, nseg = u.segreduce_u32(d, fl)
    u.check()
    want_sums, want_nseg = oracle.segreduce(a, f)
    assert int(host(nseg)[0]) == want_nseg
    assert np.array_equal(host(sums)[:want_nseg], want_sums)


@pytest.mark.parametrize("with_sums", [False, True], ids=["scan", "scan+sums"])
@pytest.mark.parametrize("kind", ["none", "regular4"])
@pytest.mark.parametrize("n,skip", [(10240 * 8 + 7, 2), ((1 << 22) + 12345, 3)], ids=["9-tiles", "411-tiles"])
def test_timeout_is_reported_and_workspace_recovers(u, n, skip, kind, with_sums):
    # Tile `skip` never publishes its two carry words: the tiles after it
    # that need them wait the given limit, give up, and the status says so;
    # the workspace then serves a normal call.
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    a, f = inputs.scan_values(n, 13), heads(kind, n, 13)
    d, fl = dev(a), dev(f)
    sums = torch.zeros(n, dtype=torch.int32, device="cuda")
    nseg = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = u.Workspace(lib.u32scan_workspace_bytes(_native.OP_SEGSCAN, n), torch.device("cuda"))
    s = torch.cuda.current_stream().cuda_stream
    rc = lib.u32scan_test_segscan_skip_publish(d.data_ptr(), fl.data_ptr(), n, sums.data_ptr() if with_sums else None,
                                               n if with_sums else 0, nseg.data_ptr(), ws.ptr, ws.nbytes, skip,
                                               20_000_000, s)
    assert rc == _native.OK
    assert lib.u32scan_check(ws.ptr, s) == _native.ETIMEOUT
    assert lib.u32scan_check(ws.ptr, s) == _native.OK  # the status was cleared
    d = dev(a)
    sums = torch.full((n,), -1, dtype=torch.int32, device="cuda") if with_sums else None
    nseg = u.segscan_inclusive_u32(d, fl, sums, workspace=ws)
    assert lib.u32scan_check(ws.ptr, s) == _native.OK
    want_sums, want_nseg = oracle.segreduce(a, f)
    assert np.array_equal(host(d), oracle.segscan_inclusive(a, f))
    assert int(host(nseg)[0]) == want_nseg
    if with_sums:
        assert np.array_equal(host(sums)[:want_nseg], want_sums)

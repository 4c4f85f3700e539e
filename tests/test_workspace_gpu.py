"""Every operation keeps the shared 256-byte workspace header (tile counter,
call epoch, device status, the segment count word) valid: interleaving all operations on one
workspace, in every order, must give oracle-exact results and a clean
status after each call."""

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


def dev32(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32).copy()).cuda()


def host_u32(t):
    return t.cpu().numpy().view(np.uint32)


def run_op(u, ws, which, n, seed):
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    if which == "scan":
        a = inputs.splitmix_u32(seed, 0, n)
        d = dev32(a)
        total = u.scan_exclusive_u32(d, workspace=ws)
        want, want_total = oracle.scan_exclusive(a)
        ok = np.array_equal(host_u32(d), want) and int(host_u32(total)[0]) == want_total
    elif which == "segscan":
        a = inputs.splitmix_u32(seed, 0, n)
        f = inputs.segment_heads_geometric(n, seed, log2_mean=6)
        d, fl = dev32(a), dev32(f)
        # with sums, or without (the segment count then goes through a
        # header word of its own)
        sums = torch.empty(n, dtype=torch.int32, device="cuda") if seed % 2 else None
        nseg = u.segscan_inclusive_u32(d, fl, sums, workspace=ws)
        want_sums, want_n = oracle.segreduce(a, f)
        ok = (np.array_equal(host_u32(d), oracle.segscan_inclusive(a, f)) and int(nseg.item()) == want_n
              and (sums is None or np.array_equal(host_u32(sums)[:want_n], want_sums)))
    elif which == "compact":
        f = inputs.compact_flags(n, seed, 0.1)
        offsets, indices, count = u.compact_indices_u32(dev32(f), workspace=ws)
        wo, wi, wc = oracle.compact_indices(f)
        ok = (np.array_equal(offsets.cpu().numpy(), wo) and np.array_equal(indices.cpu().numpy(), wi)
              and int(count.item()) == wc)
    else:
        k = inputs.radix_keys(n, seed, ties=bool(seed % 2))
        perm = u.radix_sort_perm_u32(dev32(k), workspace=ws)
        ok = np.array_equal(perm.cpu().numpy(), oracle.sort_perm(k))
    status = lib.u32scan_check(ws.ptr, torch.cuda.current_stream().cuda_stream)
    return ok, status


def test_all_operations_share_one_workspace(u):
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    sizes = [1, 5000, 70001, (1 << 22) + 3]
    need = max(lib.u32scan_workspace_bytes(op, n) for op in (1, 2, 3, 4) for n in sizes)
    ws = u.Workspace(need, torch.device("cuda"))
    order = ["scan", "radix", "segscan", "compact", "radix", "scan", "compact", "segscan", "scan", "radix"]
    rng = np.random.default_rng(12)
    for k, which in enumerate(order * 2):
        n = int(rng.choice(sizes))
        ok, status = run_op(u, ws, which, n, 30 + k)
        assert status == _native.OK, (k, which, n)
        assert ok, (k, which, n)


def test_radix_leaves_nothing_that_passes_for_tile_words(u):
    """The radix sort keeps histograms and ping-pong buffers of keys and
    indices in the workspace; with tie-heavy keys they hold small integers,
    which (two to a 64-bit word) look like tile words tagged with a small
    epoch. A fresh workspace keeps the epochs small, and each later call
    here uses a size whose tile words cover where the sort's buffers were:
    every result must still be exact."""
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    big = 1 << 25
    need = max([lib.u32scan_workspace_bytes(op, big) for op in (1, 2, 3, 6)] +
               [lib.u32scan_workspace_bytes(4, n_r) for n_r in (70001, 1 << 20)])
    # 1000 and 70001 keys: the small-sort layout (everything after the
    # header, cleared at the end); 2^20: the large-sort one (buffers past
    # the span other operations' words take, nothing cleared)
    for n_r in (1000, 70001, 1 << 20):
        for which in ("scan", "segscan", "compact", "values", "scan64"):
            ws = u.Workspace(need, torch.device("cuda"))
            k = inputs.radix_keys(n_r, 3, ties=True)
            perm = u.radix_sort_perm_u32(dev32(k), workspace=ws)
            assert np.array_equal(perm.cpu().numpy(), oracle.sort_perm(k))
            if which in ("scan", "segscan", "compact"):
                ok, status = run_op(u, ws, which, big, 5)
            elif which == "values":
                v, f = inputs.scan_values(big, 4), inputs.compact_flags(big, 4, 0.1)
                out, count = u.compact_values_u32(dev32(v), dev32(f), workspace=ws)
                want, used = oracle.compact_values(v, f, np.zeros(big, np.uint32))
                ok = int(count.item()) == used and np.array_equal(host_u32(out)[:used], want[:used])
                status = lib.u32scan_check(ws.ptr, torch.cuda.current_stream().cuda_stream)
            else:
                a = inputs.scan_values_u64(big, 5)
                d = torch.from_numpy(a.view(np.int64).copy()).cuda()
                total = u.scan_u64_op(d, "add", False, workspace=ws)
                want, want_total = oracle.scan_op_u64(a, "add", False)
                ok = np.array_equal(d.cpu().numpy().view(np.uint64), want) and \
                    int(total.cpu().numpy().view(np.uint64)[0]) == want_total
                status = lib.u32scan_check(ws.ptr, torch.cuda.current_stream().cuda_stream)
            assert status == _native.OK, (n_r, which)
            assert ok, (n_r, which)


# Header words (32-bit) of a workspace: tile counter, launch count (epoch),
# status, detail, blocks finished.
H_COUNTER, H_EPOCH, H_DONE = 0, 1, 4
TAG_PERIOD = 1 << 29  # carry-word tags repeat every 2^29 launches


def header(ws):
    return ws.buf[:256].view(torch.int32).cpu().numpy().view(np.uint32)


def set_epoch(ws, e):
    ws.buf[4 * H_EPOCH: 4 * H_EPOCH + 4].copy_(
        torch.tensor([e & 0xffffffff], dtype=torch.int64).to(torch.int32).view(torch.uint8))


def run_exact(u, ws, which, n, seed):
    """One call of `which` on ws, checked element by element against the oracle."""
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    if which in ("scan", "segscan", "compact"):
        return run_op(u, ws, which, n, seed)
    if which == "segscan_nosums":
        a, f = inputs.splitmix_u32(seed, 0, n), inputs.segment_heads_geometric(n, seed, log2_mean=6)
        d = dev32(a)
        nseg = u.segscan_inclusive_u32(d, dev32(f), workspace=ws)
        ok = (np.array_equal(host_u32(d), oracle.segscan_inclusive(a, f))
              and int(nseg.item()) == oracle.segreduce(a, f)[1])
    elif which == "values":
        v, f = inputs.scan_values(n, seed), inputs.compact_flags(n, seed, 0.9)
        out, count = u.compact_values_u32(dev32(v), dev32(f), workspace=ws)
        want, used = oracle.compact_values(v, f, np.zeros(n, np.uint32))
        ok = int(count.item()) == used and np.array_equal(host_u32(out)[:used], want[:used])
    else:  # scan64
        a = inputs.scan_values_u64(n, seed)
        d = torch.from_numpy(a.view(np.int64).copy()).cuda()
        total = u.scan_u64_op(d, "add", False, workspace=ws)
        want, want_total = oracle.scan_op_u64(a, "add", False)
        ok = np.array_equal(d.cpu().numpy().view(np.uint64), want) and \
            int(total.cpu().numpy().view(np.uint64)[0]) == want_total
    return ok, lib.u32scan_check(ws.ptr, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("which,big", [("scan", (1 << 22) + 77), ("scan", 300001), ("segscan", (1 << 22) + 5),
                                       ("segscan_nosums", (1 << 22) + 5), ("compact", (1 << 22) + 9),
                                       ("values", (1 << 22) + 9), ("scan64", (1 << 21) + 3)])
def test_tag_period_end_clears_old_carry_words(u, which, big):
    """Carry-word tags repeat every 2^29 launches on a workspace. A long call
    leaves tagged words far out; shorter calls then advance the launch count
    (here: set directly in the header) without touching those words. The
    launch that ends the tag period must zero them, or the next long call
    whose tag matches the old one would add them in as published carries."""
    from u32_prefix_scan_gb300 import _native

    op = {"scan": 1, "segscan": 2, "segscan_nosums": 2, "compact": 3, "values": 3, "scan64": 6}[which]
    ws = u.Workspace(_native.lib().u32scan_workspace_bytes(op, big), torch.device("cuda"))
    set_epoch(ws, TAG_PERIOD - 2)
    ok, status = run_exact(u, ws, which, big, 41)  # the long call: tag of launch 2^29 - 2
    assert status == _native.OK and ok
    h = header(ws)
    assert h[H_EPOCH] == TAG_PERIOD - 1 and h[H_COUNTER] == 0 and h[H_DONE] == 0
    ok, status = run_exact(u, ws, which, 1000, 42)  # launch 2^29 - 1 ends the period
    assert status == _native.OK and ok
    assert header(ws)[H_EPOCH] == TAG_PERIOD
    set_epoch(ws, 2 * TAG_PERIOD - 2)  # the same tag as the long call's
    ok, status = run_exact(u, ws, which, big, 43)
    assert status == _native.OK
    assert ok, "a carry word from the previous tag period was taken as published"
    h = header(ws)
    assert h[H_EPOCH] == 2 * TAG_PERIOD - 1 and h[H_COUNTER] == 0 and h[H_DONE] == 0


def test_tag_period_end_on_a_radix_pass_clears_other_operations_words(u):
    """The launch that ends a tag period can be a radix digit pass. A small
    sort (its buffers packed after the header) clears at the end of the
    call instead of counting its blocks out; that clear must therefore reach
    every word another operation may have left, not only the sort's own
    (smaller) part of the workspace. Here a scan of
    2^26 elements leaves tile words out to 33 KB, a sort of 1000 keys (a
    23 KB workspace part) ends the period with its first digit pass, and a
    second scan carrying the first one's tag must still be exact."""
    from u32_prefix_scan_gb300 import _native

    big = (1 << 26) + 77
    ws = u.Workspace(_native.lib().u32scan_workspace_bytes(1, big), torch.device("cuda"))
    assert _native.lib().u32scan_workspace_bytes(4, 1000) < ws.nbytes
    set_epoch(ws, TAG_PERIOD - 2)
    ok, status = run_op(u, ws, "scan", big, 51)  # tag of launch 2^29 - 2
    assert status == _native.OK and ok
    assert header(ws)[H_EPOCH] == TAG_PERIOD - 1
    k = inputs.radix_keys(1000, 52)  # four active digit passes; the first ends the period
    perm = u.radix_sort_perm_u32(dev32(k), workspace=ws)
    assert np.array_equal(perm.cpu().numpy(), oracle.sort_perm(k))
    assert header(ws)[H_EPOCH] == TAG_PERIOD + 3
    set_epoch(ws, 2 * TAG_PERIOD - 2)  # the first scan's tag again
    ok, status = run_op(u, ws, "scan", big, 53)
    assert status == _native.OK
    assert ok, "a scan's carry word from the ended tag period was taken as published"


def test_tag_period_end_on_a_large_radix_pass(u):
    """A large sort keeps its buffers past the span other operations' carry
    words can take and clears nothing at its end. When its first digit pass
    ends a tag period, that pass's blocks count themselves out and the last
    one zeroes the span: a later scan carrying an earlier scan's tag must
    still be exact, and so must the sort's own later passes (new period)."""
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    big, n_r = (1 << 26) + 77, 1 << 20
    ws = u.Workspace(max(lib.u32scan_workspace_bytes(1, big), lib.u32scan_workspace_bytes(4, n_r)),
                     torch.device("cuda"))
    set_epoch(ws, TAG_PERIOD - 2)
    ok, status = run_op(u, ws, "scan", big, 61)  # tag of launch 2^29 - 2
    assert status == _native.OK and ok
    assert header(ws)[H_EPOCH] == TAG_PERIOD - 1
    k = inputs.radix_keys(n_r, 62)  # four active digit passes; the first ends the period
    perm = u.radix_sort_perm_u32(dev32(k), workspace=ws)
    assert lib.u32scan_check(ws.ptr, torch.cuda.current_stream().cuda_stream) == _native.OK
    assert np.array_equal(perm.cpu().numpy(), oracle.sort_perm(k))
    h = header(ws)
    assert h[H_EPOCH] == TAG_PERIOD + 3 and h[H_COUNTER] == 0 and h[H_DONE] == 0
    set_epoch(ws, 2 * TAG_PERIOD - 2)  # the first scan's tag again
    ok, status = run_op(u, ws, "scan", big, 63)
    assert status == _native.OK
    assert ok, "a scan's carry word from the ended tag period was taken as published"


def test_large_radix_clears_its_carry_words_past_the_shared_span(u):
    """A sort of more than 4096 tiles (here 3 x 2^24 keys) has carry words
    past the span other operations' words can take, where another call's
    histograms or buffers may lie. Words planted there that read as
    published inclusive zeros carrying the sort's first tag (every slot
    computed from them would stay in bounds, only wrong) must be cleared
    before the passes run."""
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    n = 3 << 24
    reach = max(lib.u32scan_workspace_bytes(op, (1 << 32) - 1) for op in (1, 2, 3, 6))
    reach = (reach + 255) // 256 * 256
    n_tiles = (n + 11263) // 11264
    desc_end = 256 + (8 * 256 * n_tiles + 255) // 256 * 256
    assert desc_end > reach
    ws = u.Workspace(lib.u32scan_workspace_bytes(4, n), torch.device("cuda"))
    e = int(header(ws)[H_EPOCH])
    word = (((e & (TAG_PERIOD - 1)) + 1) << 34) | (1 << 32)  # tag of the first pass, inclusive, count 0
    planted = torch.full(((desc_end - reach) // 8,), word, dtype=torch.int64, device="cuda")
    ws.buf[reach:desc_end].copy_(planted.view(torch.uint8))
    k = inputs.radix_keys(n, 72)
    perm = u.radix_sort_perm_u32(dev32(k), workspace=ws)
    assert lib.u32scan_check(ws.ptr, torch.cuda.current_stream().cuda_stream) == _native.OK
    assert np.array_equal(perm.cpu().numpy(), oracle.sort_perm(k))


def test_reduce_leaves_no_partials_that_pass_for_tile_words(u):
    """count_nonzero_u32 and reduce_u32_op fold per-block partials in the
    workspace, where a scan keeps its tile words. Left behind, two partials
    side by side read as one 64-bit word whose tag field is a partial's bits:
    at the launch count that tag names, a scan would take the word for a
    published carry. The reduce must leave that region zero. End to end: the
    word left at the scan's tile 0 (if any) sets the launch count its tag
    names, tile 0 of a scan is made never to publish (the test hook), and
    tile 1 must then wait for it and time out rather than take the word."""
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    n = 1 << 20
    ws = u.Workspace(max(lib.u32scan_workspace_bytes(_native.OP_SCAN, n),
                         lib.u32scan_workspace_bytes(_native.OP_REDUCE, n)), torch.device("cuda"))
    span = lib.u32scan_workspace_bytes(_native.OP_REDUCE, n)
    ones = torch.ones(16384, dtype=torch.int32, device="cuda")
    assert int(u.count_nonzero_u32(ones, workspace=ws).item()) == 16384
    word = int(ws.buf[256:264].cpu().numpy().view(np.uint64)[0])
    set_epoch(ws, (word >> 34) - 1 if word >> 34 else 1535)  # the launch count a left word's tag would name
    a = inputs.scan_values(n, 61)
    d, total = dev32(a), torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.u32scan_test_scan_skip_publish(d.data_ptr(), n, total.data_ptr(), ws.ptr, ws.nbytes, 0,
                                              20_000_000, stream) == _native.OK
    assert lib.u32scan_check(ws.ptr, stream) == _native.ETIMEOUT, "a stale partial was taken as tile 0's carry"
    # the workspace serves a normal call afterwards
    d = dev32(a)
    total = u.scan_exclusive_u32(d, workspace=ws)
    assert lib.u32scan_check(ws.ptr, stream) == _native.OK
    want, want_total = oracle.scan_exclusive(a)
    assert np.array_equal(host_u32(d), want) and int(host_u32(total)[0]) == want_total
    # and directly: after either fold on a zero-filled workspace, the span is zero again
    for fold in (lambda: u.count_nonzero_u32(ones, workspace=ws), lambda: u.reduce_u32_op(ones, "add", workspace=ws)):
        ws.buf.zero_()
        assert int(fold().item()) == 16384
        assert not ws.buf[256:span].any(), "a fold left its partials in the workspace"


def test_host_scan_leaves_nothing_that_passes_for_tile_words(u):
    """scan_exclusive_u32_host stages its chunks in the workspace, past the
    chunk scan's own tile words and inside the span where other operations
    keep theirs; the scanned chunks (increasing integers here) read, two
    side by side, as words whose tag field names some launch count. The
    word left at tile t of a later scan sets that launch count, tile t is
    made never to publish (the test hook), and tile t + 1 must then wait
    for it and time out rather than take the staged data for its carry."""
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    n_host, n = 1 << 22, 1 << 26
    ws = u.Workspace(max(lib.u32scan_workspace_bytes(_native.OP_SCAN_HOST, n_host),
                         lib.u32scan_workspace_bytes(_native.OP_SCAN, n)), torch.device("cuda"))
    host_in = torch.ones(n_host, dtype=torch.int32).pin_memory()
    out, total = u.scan_exclusive_u32_host(host_in, workspace=ws)
    torch.cuda.synchronize()
    assert int(total[0]) == n_host and int(out[-1]) == n_host - 1
    n_tiles = (lib.u32scan_workspace_bytes(_native.OP_SCAN, n) - 256) // 8  # at least the scan's tiles
    t = 3000  # a tile word 24 KB in, among the host scan's staging slots
    assert t + 2 < n_tiles - 32
    word = int(ws.buf[256 + 8 * t: 264 + 8 * t].cpu().numpy().view(np.uint64)[0])
    set_epoch(ws, (word >> 34) - 1 if word >> 34 else 1535)  # the launch count a left word's tag would name
    a = inputs.scan_values(n, 62)
    d, tot = dev32(a), torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.u32scan_test_scan_skip_publish(d.data_ptr(), n, tot.data_ptr(), ws.ptr, ws.nbytes, t,
                                              20_000_000, stream) == _native.OK
    assert lib.u32scan_check(ws.ptr, stream) == _native.ETIMEOUT, "staged host data was taken as a carry"
    d = dev32(a)
    tot = u.scan_exclusive_u32(d, workspace=ws)
    assert lib.u32scan_check(ws.ptr, stream) == _native.OK
    want, want_total = oracle.scan_exclusive(a)
    assert np.array_equal(host_u32(d), want) and int(host_u32(tot)[0]) == want_total

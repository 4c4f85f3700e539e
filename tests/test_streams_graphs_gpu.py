"""Concurrent calls on separate streams, and calls captured in CUDA graphs,
against the CPU oracle, through the C ABI.

Streams: calls on different streams with their own workspaces run
concurrently and each gives the oracle's result. Graphs: a call captured once
(with a workspace allocated and zero-filled beforehand) and replayed many
times rescans whatever the captured buffers hold at each replay; every
replay is checked bit for bit. The radix sort's memsets and its seven
launches, and the segmented and compaction kernels, capture the same way.
"""

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


def dev32(a: np.ndarray):
    return torch.from_numpy(a.view(np.int32).copy()).cuda()


def host32(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def workspace(u, op, n):
    from u32_prefix_scan_gb300 import _native

    return u.Workspace(_native.lib().u32scan_workspace_bytes(op, n), torch.device("cuda", torch.cuda.current_device()))


def test_concurrent_scans_on_four_streams(u):
    from u32_prefix_scan_gb300 import _native

    sizes = [(1 << 22) + 5, (1 << 24) + 77, 100003, (1 << 23) + 1]
    streams = [torch.cuda.Stream() for _ in sizes]
    host = [inputs.scan_values(n, 20 + i) for i, n in enumerate(sizes)]
    data = [dev32(a) for a in host]
    wss = [workspace(u, _native.OP_SCAN, n) for n in sizes]
    totals = []
    torch.cuda.synchronize()
    for _ in range(3):  # repeated, so that the streams' calls overlap
        for i, (s, d, ws) in enumerate(zip(streams, data, wss)):
            d.copy_(torch.from_numpy(host[i].view(np.int32)).cuda())
        torch.cuda.synchronize()
        totals = []
        for i, (s, d, ws) in enumerate(zip(streams, data, wss)):
            with torch.cuda.stream(s):
                fn = u.scan_inclusive_u32 if i % 2 else u.scan_exclusive_u32
                totals.append(fn(d, stream=s, workspace=ws))
        torch.cuda.synchronize()
        for i, (d, ws) in enumerate(zip(data, wss)):
            u.check(stream=streams[i], workspace=ws)
            want, want_total = (oracle.scan_inclusive if i % 2 else oracle.scan_exclusive)(host[i])
            assert np.array_equal(host32(d), want)
            assert int(host32(totals[i])[0]) == want_total


def test_concurrent_primitives_on_separate_streams(u):
    from u32_prefix_scan_gb300 import _native

    n = (1 << 22) + 333
    vals, keys = inputs.scan_values(n, 31), inputs.radix_keys(n, 32)
    heads = inputs.segment_heads_geometric(n, 33)
    flags = (inputs.splitmix_u32(34, 1, n) < np.uint32(1 << 30)).astype(np.int32)
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    d_v, d_h = dev32(vals), torch.from_numpy(heads).cuda()
    d_f, d_k = torch.from_numpy(flags).cuda(), dev32(keys)
    perm = torch.empty(n, dtype=torch.int32, device="cuda")
    ws1, ws2, ws3 = (workspace(u, _native.OP_SEGSCAN, n), workspace(u, _native.OP_COMPACT, n),
                     workspace(u, _native.OP_RADIX, n))
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        nseg = u.segscan_inclusive_u32(d_v, d_h, stream=s1, workspace=ws1)
    with torch.cuda.stream(s2):
        offsets, indices, count = u.compact_indices_u32(d_f, stream=s2, workspace=ws2)
    with torch.cuda.stream(s3):
        u.radix_sort_perm_u32(d_k, perm, stream=s3, workspace=ws3)
    torch.cuda.synchronize()
    assert np.array_equal(host32(d_v), oracle.segscan_inclusive(vals, heads))
    assert int(host32(nseg)[0]) == oracle.segreduce(vals, heads)[1]
    want_off, want_idx, want_count = oracle.compact_indices(flags)
    assert np.array_equal(offsets.cpu().numpy(), want_off)
    assert np.array_equal(indices.cpu().numpy(), want_idx)
    assert int(count[0]) == want_count
    assert np.array_equal(perm.cpu().numpy(), oracle.sort_perm(keys))


@pytest.mark.parametrize("n", [1 << 16, (1 << 22) + 7])  # the one-tile-per-block and the persistent kernel
def test_scan_replayed_from_a_cuda_graph(u, n):
    from u32_prefix_scan_gb300 import _native

    d = torch.empty(n, dtype=torch.int32, device="cuda")
    total = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = workspace(u, _native.OP_SCAN, n)
    d.copy_(dev32(inputs.scan_values(n, 40)))
    u.scan_exclusive_u32(d, total, workspace=ws)  # first call outside the capture (per-device set-up)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            u.scan_exclusive_u32(d, total, stream=s, workspace=ws)
    for rep in range(5):
        a = inputs.scan_values(n, 41 + rep)
        d.copy_(dev32(a))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        want, want_total = oracle.scan_exclusive(a)
        assert np.array_equal(host32(d), want), rep
        assert int(host32(total)[0]) == want_total
    u.check(stream=s, workspace=ws)


def test_primitives_replayed_from_cuda_graphs(u):
    from u32_prefix_scan_gb300 import _native

    n = (1 << 21) + 99
    d_v = torch.empty(n, dtype=torch.int32, device="cuda")
    d_h = torch.empty(n, dtype=torch.int32, device="cuda")
    d_f = torch.empty(n, dtype=torch.int32, device="cuda")
    d_k = torch.empty(n, dtype=torch.int32, device="cuda")
    perm = torch.empty(n, dtype=torch.int32, device="cuda")
    offsets = torch.empty(n, dtype=torch.int32, device="cuda")
    indices = torch.empty(n, dtype=torch.int32, device="cuda")
    count = torch.empty(1, dtype=torch.int32, device="cuda")
    nseg = torch.empty(1, dtype=torch.int32, device="cuda")
    ws1, ws2, ws3 = (workspace(u, _native.OP_SEGSCAN, n), workspace(u, _native.OP_COMPACT, n),
                     workspace(u, _native.OP_RADIX, n))

    def fill(seed):
        vals, keys = inputs.scan_values(n, seed), inputs.radix_keys(n, seed + 1, ties=seed % 2 == 1)
        heads = inputs.segment_heads_regular(n, 4) if seed % 2 else inputs.segment_heads_geometric(n, seed + 2)
        flags = (inputs.splitmix_u32(seed + 3, 1, n) < np.uint32(3 << 30)).astype(np.int32)
        d_v.copy_(dev32(vals))
        d_h.copy_(torch.from_numpy(heads).cuda())
        d_f.copy_(torch.from_numpy(flags).cuda())
        d_k.copy_(dev32(keys))
        return vals, heads, flags, keys

    def calls(s):
        u.segscan_inclusive_u32(d_v, d_h, None, nseg, stream=s, workspace=ws1)
        u.compact_indices_u32(d_f, offsets, indices, count, stream=s, workspace=ws2)
        u.radix_sort_perm_u32(d_k, perm, stream=s, workspace=ws3)

    fill(50)
    calls(torch.cuda.current_stream())  # first calls outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            calls(s)
    for rep in range(4):
        vals, heads, flags, keys = fill(51 + rep)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host32(d_v), oracle.segscan_inclusive(vals, heads)), rep
        assert int(host32(nseg)[0]) == oracle.segreduce(vals, heads)[1]
        want_off, want_idx, want_count = oracle.compact_indices(flags)
        assert np.array_equal(offsets.cpu().numpy(), want_off)
        assert np.array_equal(indices.cpu().numpy(), want_idx)
        assert int(count[0]) == want_count
        assert np.array_equal(perm.cpu().numpy(), oracle.sort_perm(keys))

"""GPU runs at the largest sizes each entry point accepts, through the C ABI.

Element counts up to 2^32 - 1 (scans, u64 scans, segmented scans) and
2^31 - 1 (compaction, radix sort: int32 outputs), and a host-buffer scan
past 2^32. The inputs are structured so that every result has a closed
form (all-ones scans are the index sequence; a third of the flags kept at
every third index; strictly decreasing keys sort into the reversed index
order), checked element by element on the device in chunks. What they pin
is the index arithmetic past 2^31 and near the limits: tile numbers, byte
offsets, the compaction's tail and the wrapped totals.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

M32 = 1 << 32
CHUNK = 1 << 28


@pytest.fixture(scope="module")
def u():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import build

    build.build()
    import u32_prefix_scan_gb300 as u

    yield u
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(autouse=True)
def _release():
    yield
    # drop the cached per-stream workspaces (a 2^31-key sort's is 24 GB) and
    # the caching allocator's blocks, so later tests start from a light GPU
    from u32_prefix_scan_gb300 import api

    torch.cuda.synchronize()
    api.Workspace._cache.clear()
    torch.cuda.empty_cache()


def as_u32(t):
    """int64 view of int32 bits, read as unsigned."""
    return t.to(torch.int64) & 0xFFFFFFFF


def check_chunks(t, expect, n):
    """t[s:e] (as unsigned 32-bit) equals expect(arange(s, e)) for every chunk."""
    for s in range(0, n, CHUNK):
        e = min(n, s + CHUNK)
        idx = torch.arange(s, e, dtype=torch.int64, device=t.device)
        assert torch.equal(as_u32(t[s:e]), expect(idx)), f"mismatch in [{s}, {e})"


@pytest.mark.parametrize("inclusive", [False, True])
def test_scan_at_2_32_minus_1(u, inclusive):
    n = M32 - 1
    d = torch.ones(n, dtype=torch.int32, device="cuda")
    total = (u.scan_inclusive_u32 if inclusive else u.scan_exclusive_u32)(d)
    u.check()
    check_chunks(d, (lambda i: (i + 1) & 0xFFFFFFFF) if inclusive else (lambda i: i & 0xFFFFFFFF), n)
    assert int(as_u32(total)[0]) == n % M32


def test_u64_scan_at_2_32_minus_1(u):
    n = M32 - 1
    d = torch.ones(n, dtype=torch.int64, device="cuda")
    total = u.scan_u64_op(d, "add", inclusive=False)
    u.check()
    for s in range(0, n, CHUNK):
        e = min(n, s + CHUNK)
        assert torch.equal(d[s:e], torch.arange(s, e, dtype=torch.int64, device="cuda"))
    assert int(total[0]) == n


def test_segscan_at_2_32_minus_1(u):
    n = M32 - 1
    h1 = 3_000_000_017  # a head past 2^31
    d = torch.ones(n, dtype=torch.int32, device="cuda")
    f = torch.zeros(n, dtype=torch.int32, device="cuda")
    f[h1] = 5
    sums = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    nseg = u.segscan_inclusive_u32(d, f, sums)
    u.check()
    check_chunks(d, lambda i: torch.where(i < h1, i + 1, i - h1 + 1), n)
    assert int(nseg[0]) == 2
    assert [int(x) for x in as_u32(sums[:2])] == [h1, n - h1]
    assert int(sums[2]) == -1


def test_compact_at_2_31_minus_1(u):
    n = (1 << 31) - 1
    flags = (torch.arange(n, dtype=torch.int64, device="cuda") % 3 == 0).to(torch.int32)
    offsets, indices, count = u.compact_indices_u32(flags)
    u.check()
    del flags
    kept = (n + 2) // 3
    assert int(count[0]) == kept
    check_chunks(offsets, lambda i: i // 3 + 1, n)
    check_chunks(indices, lambda i: torch.where(i < kept, 3 * i, torch.full_like(i, 0xFFFFFFFF)), n)


def test_radix_perm_at_2_31_minus_1(u):
    n = (1 << 31) - 1
    keys = torch.arange(n - 1, -1, -1, dtype=torch.int64, device="cuda").to(torch.int32)  # strictly decreasing
    perm = torch.empty(n, dtype=torch.int32, device="cuda")
    u.radix_sort_perm_u32(keys, perm)
    u.check()
    check_chunks(perm, lambda i: n - 1 - i, n)


def test_host_scan_past_2_32(u):
    n = M32 + (1 << 23) + 5  # the chunk chain crosses 2^32 elements
    h = torch.ones(n, dtype=torch.int32).pin_memory()
    _, total = u.scan_exclusive_u32_host(h, h)
    torch.cuda.synchronize()
    a = h.numpy().view(np.uint32)
    for s in range(0, n, CHUNK):
        e = min(n, s + CHUNK)
        assert np.array_equal(a[s:e], (np.arange(s, e, dtype=np.uint64) & 0xFFFFFFFF).astype(np.uint32)), s
    assert int(total.numpy().view(np.uint32)[0]) == n % M32

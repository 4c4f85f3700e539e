"""GPU parity of the host-buffer scans (scan_exclusive_u32_host,
scan_inclusive_u32_host) against the CPU oracle, through the C ABI.

The array is pinned host memory; the library moves it through device
staging slots in chunks, each chunk's scan starting from the sum of the
chunks before it. Bit-exact, element by element: one chunk and many, ragged
last chunks, more chunks than staging slots (the ring wraps), in place and
into a second buffer, a side stream, repeated calls on one workspace, the
empty array, the full 2^28 workload, and the rejection of pageable memory.
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


def pinned(a: np.ndarray):
    t = torch.empty(a.size, dtype=torch.int32).pin_memory()
    t.numpy()[:] = a.view(np.int32)
    return t


def as_u32(t) -> np.ndarray:
    return t.numpy().view(np.uint32)


def want(inclusive, a):
    return (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(a)


# one chunk; 2^18-element chunks (2, 5 and 9 of them: the 4-slot ring wraps);
# eight chunks just over 2^22 elements with a last one just under (the
# persistent and the one-tile-per-block kernels)
SIZES = [1, 2, 5, 1000, (1 << 18) - 3, (1 << 18) + 7, 5 * (1 << 18) - 1, (1 << 21) + 12345,
         (1 << 25) + 777]


@pytest.mark.parametrize("inclusive", [False, True])
@pytest.mark.parametrize("n", SIZES)
def test_parity_sizes(u, inclusive, n):
    a = inputs.scan_values(n, 11)
    h_in = pinned(a)
    fn = u.scan_inclusive_u32_host if inclusive else u.scan_exclusive_u32_host
    h_out, total = fn(h_in)
    torch.cuda.synchronize()
    w, wt = want(inclusive, a)
    assert np.array_equal(as_u32(h_out), w)
    assert int(as_u32(total)[0]) == wt
    assert np.array_equal(as_u32(h_in), a)  # the input is only read


@pytest.mark.parametrize("inclusive", [False, True])
def test_in_place_on_a_side_stream(u, inclusive):
    n = 3 * (1 << 22) + 5
    a = inputs.scan_values(n, 12)
    h = pinned(a)
    s = torch.cuda.Stream()
    fn = u.scan_inclusive_u32_host if inclusive else u.scan_exclusive_u32_host
    out, total = fn(h, h, stream=s)
    assert out is h
    s.synchronize()
    u.check(stream=s)
    w, wt = want(inclusive, a)
    assert np.array_equal(as_u32(h), w)
    assert int(as_u32(total)[0]) == wt


def test_repeated_calls_share_one_workspace(u):
    # the same workspace serves calls of different lengths, in stream order
    ws = u.Workspace(1 << 27, torch.device("cuda", 0))
    for n, seed in (((1 << 21) + 3, 13), (1000, 14), ((1 << 23) + 99, 15), ((1 << 21) + 3, 16)):
        a = inputs.scan_values(n, seed)
        h_out, total = u.scan_exclusive_u32_host(pinned(a), workspace=ws)
        torch.cuda.synchronize()
        w, wt = oracle.scan_exclusive(a)
        assert np.array_equal(as_u32(h_out), w)
        assert int(as_u32(total)[0]) == wt
    u.check(workspace=ws)


def test_small_values_total_is_the_exact_sum(u):
    n = (1 << 24) + 1
    a = inputs.scan_values(n, 2) >> 28
    _, total = u.scan_inclusive_u32_host(pinned(a))
    torch.cuda.synchronize()
    assert int(as_u32(total)[0]) == int(a.astype(np.uint64).sum())


def test_empty_writes_zero_total(u):
    h = torch.empty(0, dtype=torch.int32).pin_memory()
    total = torch.full((1,), 77, dtype=torch.int32).pin_memory()
    u.scan_exclusive_u32_host(h, h, total)
    torch.cuda.synchronize()
    assert int(total[0]) == 0


def test_pageable_memory_is_rejected(u):
    from u32_prefix_scan_gb300 import _native

    a = torch.zeros(1000, dtype=torch.int32)  # not pinned
    out = torch.empty(1000, dtype=torch.int32).pin_memory()
    ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_SCAN_HOST, 1000), torch.device("cuda", 0))
    rc = _native.lib().scan_exclusive_u32_host(a.data_ptr(), out.data_ptr(), 1000, None, ws.ptr, ws.nbytes, None)
    assert rc == _native.EINVAL
    with pytest.raises(ValueError, match="pinned"):
        u.scan_exclusive_u32_host(a)


def test_full_workload_2_28(u):
    n = 1 << 28
    a = inputs.scan_values(n, 2)
    h = pinned(a)
    _, total = u.scan_exclusive_u32_host(h, h)
    torch.cuda.synchronize()
    w, wt = oracle.scan_exclusive(a)
    assert np.array_equal(as_u32(h), w)
    assert int(as_u32(total)[0]) == wt

"""GPU parity of the U32 scans against the CPU oracle, through the C ABI.

Bit-exact, element by element: sizes from empty through several tiles of
both launch shapes with ragged tails, every 4-byte misalignment, repeated
calls on one workspace, the two benchmark workloads (2^16 and 2^28), the
small-value variant, closed forms at full size, and the bounded carry wait.
"""

import numpy as np
import pytest

import oracle
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

M32 = 1 << 32


@pytest.fixture(scope="module")
def u():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import build

    build.build()
    import u32_prefix_scan_gb300 as u

    return u


def to_dev(a: np.ndarray, offset: int = 0):
    """Device int32 view of a uint32 array, starting `offset` elements into
    a larger allocation (to exercise misaligned starts)."""
    buf = torch.empty(a.size + offset + 4, dtype=torch.int32, device="cuda")
    view = buf[offset: offset + a.size]
    view.copy_(torch.from_numpy(a.view(np.int32)))
    return view


def to_host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def run(u, inclusive, a, offset=0):
    d = to_dev(a, offset)
    fn = u.scan_inclusive_u32 if inclusive else u.scan_exclusive_u32
    total = fn(d)
    u.check()
    return to_host(d), int(to_host(total)[0])


SIZES = [1, 2, 3, 4, 5, 31, 32, 33, 127, 1000, 2047, 2048, 2049, 3 * 2048 + 77, 8192 * 5 + 3,
         65536, 65536 + 1, (1 << 19) - 1, 1 << 19, (1 << 19) + 1, (1 << 22) - 1, 1 << 22, (1 << 22) + 1,
         3 * 16384 * 100 + 12345]


@pytest.mark.parametrize("inclusive", [False, True])
@pytest.mark.parametrize("n", SIZES)
def test_parity_sizes(u, inclusive, n):
    a = inputs.scan_values(n, 1)
    got, total = run(u, inclusive, a)
    want, want_total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(a)
    assert np.array_equal(got, want)
    assert total == want_total


@pytest.mark.parametrize("inclusive", [False, True])
@pytest.mark.parametrize("offset", [1, 2, 3])
@pytest.mark.parametrize("n", [5, 2049, 65536 + 7, (1 << 19) + 5, (1 << 22) + 5])
def test_parity_misaligned_start(u, inclusive, offset, n):
    a = inputs.scan_values(n, 7)
    got, total = run(u, inclusive, a, offset)
    want, want_total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(a)
    assert np.array_equal(got, want)
    assert total == want_total


def test_empty_writes_zero_total(u):
    d = torch.empty(0, dtype=torch.int32, device="cuda")
    total = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    u.scan_exclusive_u32(d, total)
    u.check()
    assert int(total.item()) == 0


def test_repeated_calls_share_one_workspace(u):
    # The workspace is never cleared between calls: stale carries of earlier
    # calls (other sizes, other forms) must never be taken for current ones.
    ws = u.Workspace(1 << 20, torch.device("cuda"))
    rng = np.random.default_rng(3)
    for k in range(40):
        n = int(rng.choice([1, 777, 2048 * 3, 65536, (1 << 22) + 3, 2048 * 40 + 1]))
        a = inputs.splitmix_u32(9, 0, n, start=k * 1000)
        inclusive = bool(k % 2)
        d = to_dev(a)
        fn = u.scan_inclusive_u32 if inclusive else u.scan_exclusive_u32
        total = fn(d, workspace=ws)
        u.check(workspace=ws)
        want, want_total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(a)
        assert np.array_equal(to_host(d), want), (k, n)
        assert int(to_host(total)[0]) == want_total


def test_workload_2_16_uniform(u):
    a = inputs.scan_values(1 << 16, 1)
    for inclusive in (False, True):
        got, total = run(u, inclusive, a)
        want, want_total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(a)
        assert np.array_equal(got, want) and total == want_total


@pytest.mark.parametrize("small", [False, True])
def test_workload_2_28_full_parity(u, small):
    # The benchmark's configuration, in the launch shape the benchmark times.
    n = 1 << 28
    a = inputs.scan_values(n, 2, small=small)
    for inclusive in (False, True):
        got, total = run(u, inclusive, a)
        want, want_total = (oracle.scan_inclusive if inclusive else oracle.scan_exclusive)(a)
        assert np.array_equal(got, want)
        assert total == want_total
        if small:
            assert total == int(a.astype(np.uint64).sum())  # no wrap below 15 * 2^28


def test_closed_forms_at_full_size(u):
    n = 1 << 28
    d = torch.ones(n, dtype=torch.int32, device="cuda")
    total = u.scan_exclusive_u32(d)
    u.check()
    assert int(total.item()) == n
    idx = torch.arange(n, dtype=torch.int64, device="cuda")
    assert torch.equal(d, idx.to(torch.int32))
    # a[i] = i: inclusive gives j(j+1)/2 mod 2^32 (wraps many times)
    d = idx.to(torch.int32)
    u.scan_inclusive_u32(d)
    u.check()
    want = ((idx * (idx + 1) // 2) % M32).to(torch.int64)
    got = d.to(torch.int64) % M32
    assert torch.equal(got, want)


@pytest.mark.parametrize("n,skip", [(2048 * 8, 2), ((1 << 22) + 4096 * 3 + 5, 3)],
                         ids=["one-tile-kernel", "persistent-kernel"])
def test_timeout_is_reported_and_workspace_recovers(u, n, skip):
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    a = inputs.scan_values(n, 11)
    d = to_dev(a)
    total = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = u.Workspace(lib.u32scan_workspace_bytes(_native.OP_SCAN, n), torch.device("cuda"))
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.u32scan_test_scan_skip_publish(d.data_ptr(), n, total.data_ptr(), ws.ptr, ws.nbytes, skip,
                                            20_000_000, stream)
    assert rc == _native.OK
    assert lib.u32scan_check(ws.ptr, stream) == _native.ETIMEOUT
    assert lib.u32scan_check(ws.ptr, stream) == _native.OK  # the status was cleared
    # the same workspace serves a normal call afterwards
    d = to_dev(a)
    total = u.scan_exclusive_u32(d, workspace=ws)
    assert lib.u32scan_check(ws.ptr, stream) == _native.OK
    want, want_total = oracle.scan_exclusive(a)
    assert np.array_equal(to_host(d), want) and int(to_host(total)[0]) == want_total

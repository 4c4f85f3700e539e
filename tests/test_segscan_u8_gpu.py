"""GPU parity of the segmented scan and reduce with one byte per head flag
(the _u8heads entry points) against the CPU oracle, through the C ABI:
byte values that test every bit position of a flag byte, every segment-
length mix of the int32 tests, flag rows at every byte offset against the
values (bulk-copied and plain-load paths), and the benchmark workloads at
full size (n = 2^26)."""

import numpy as np
import pytest

import oracle
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BYTES = np.array([1, 0x80, 0xFF, 0x10, 0x02, 0x40, 0x7F, 0x08], dtype=np.uint8)


@pytest.fixture(scope="module")
def u():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import build

    build.build()
    import u32_prefix_scan_gb300 as u

    return u


def heads8(kind: str, n: int, seed: int = 3) -> np.ndarray:
    """Byte head flags: where the pattern has a head, one of BYTES (cycled)."""
    if kind == "geometric":
        h = inputs.segment_heads_geometric(n, seed)
    elif kind == "geometric16":
        h = inputs.segment_heads_geometric(n, seed, log2_mean=4)
    elif kind == "regular4":
        h = inputs.segment_heads_regular(n, 4)
    elif kind == "all":
        h = np.ones(n, np.int32)
    elif kind == "none":
        h = np.zeros(n, np.int32)
    elif kind == "half":
        h = (inputs.splitmix_u32(seed, 1, n) < np.uint32(1 << 31)).astype(np.int32)
    else:
        raise ValueError(kind)
    return np.where(h != 0, BYTES[np.arange(n) % BYTES.size], 0).astype(np.uint8)


def dev32(a: np.ndarray, offset: int = 0):
    buf = torch.empty(a.size + offset + 4, dtype=torch.int32, device="cuda")
    view = buf[offset: offset + a.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int32)))
    return view


def dev8(f: np.ndarray, offset: int = 0):
    buf = torch.full((f.size + offset + 16,), 0x55, dtype=torch.uint8, device="cuda")
    view = buf[offset: offset + f.size]
    view.copy_(torch.from_numpy(f))
    return view


def host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def check(u, a, f, off_a=0, off_f=0, cap=None):
    n = a.size
    d, fl = dev32(a, off_a), dev8(f, off_f)
    want_sums, want_nseg = oracle.segreduce(a, f)
    cap = max(n, 1) if cap is None else cap
    sums = torch.full((max(cap, 1),), -1, dtype=torch.int32, device="cuda")
    nseg = u.segscan_inclusive_u32(d, fl, sums[:cap] if cap else None)
    u.check()
    assert np.array_equal(host(d), oracle.segscan_inclusive(a, f))
    assert int(host(nseg)[0]) == want_nseg
    k = min(cap, want_nseg)
    assert np.array_equal(host(sums)[:k], want_sums[:k])
    assert np.all(host(sums)[k:cap] == 0xFFFFFFFF)
    d3 = dev32(a, off_a)  # the form without sums, on the same input
    c3 = u.segscan_inclusive_u32(d3, fl)
    u.check()
    assert np.array_equal(host(d3), host(d)) and int(host(c3)[0]) == want_nseg
    d2 = dev32(a, off_a)
    s2, c2 = u.segreduce_u32(d2, fl)
    u.check()
    assert int(host(c2)[0]) == want_nseg and np.array_equal(host(s2)[:want_nseg], want_sums)
    assert np.array_equal(host(d2), a)


def test_byte_flags_equal_int32_flags_bitwise(u):
    # every byte value is a head exactly when non-zero
    n = 256 * 64
    a = inputs.scan_values(n, 4)
    f = np.tile(np.arange(256, dtype=np.uint8), 64)
    check(u, a, f)


SIZES = [1, 2, 5, 4096 + 3, 14336, 14336 + 1, 3 * 14336 + 77, 100003, (1 << 20) + 5]


@pytest.mark.parametrize("kind", ["geometric", "geometric16", "regular4", "all", "none", "half"])
@pytest.mark.parametrize("n", SIZES)
def test_parity(u, kind, n):
    check(u, inputs.scan_values(n, 3), heads8(kind, n))


@pytest.mark.parametrize("off_a", [0, 1, 3])
@pytest.mark.parametrize("off_f", [0, 1, 2, 3, 4, 7, 12, 15])
def test_flag_offsets(u, off_a, off_f):
    n = 3 * 14336 + 999
    check(u, inputs.scan_values(n, 6), heads8("geometric16", n, 6), off_a, off_f)


def test_capacity_below_count(u):
    n = 100003
    check(u, inputs.scan_values(n, 3), heads8("geometric16", n), cap=777)


@pytest.mark.parametrize("kind", ["geometric", "regular4"])
def test_workload_2_26_full_parity(u, kind):
    n = 1 << 26
    check(u, inputs.scan_values(n, 3), heads8(kind, n))

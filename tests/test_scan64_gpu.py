"""GPU parity of the u64 scans (every CAIRN integer operator, exclusive and
inclusive, add and mul wrapping at 2^64) against the CPU oracle, through
the C ABI: sizes across both tile shapes with ragged tails, a row starting
8 bytes past a 16-byte boundary, sums that pass 2^64, repeated calls on one
workspace, and the full benchmark row (n = 2^27)."""

import numpy as np
import pytest

import oracle
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OPS = ["add", "mul", "and", "or", "xor", "min", "max"]


@pytest.fixture(scope="module")
def u():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import build

    build.build()
    import u32_prefix_scan_gb300 as u

    return u


def dev(a: np.ndarray, offset: int = 0):
    buf = torch.empty(a.size + offset + 2, dtype=torch.int64, device="cuda")
    view = buf[offset: offset + a.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int64)))
    return view


def host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


def values(op: str, n: int, seed: int) -> np.ndarray:
    a = inputs.scan_values_u64(n, seed)
    if op == "mul":
        a = a | np.uint64(1)
    if op in ("and", "or"):  # keep the scan from saturating at once
        a = a | (np.uint64(1) << np.uint64(63)) if op == "and" else a & np.uint64(0x0101010101010101)
    return a


def check(u, a, op, inclusive, offset=0, ws=None):
    d = dev(a, offset)
    total = u.scan_u64_op(d, op, inclusive, workspace=ws)
    u.check(workspace=ws)
    want, want_total = oracle.scan_op_u64(a, op, inclusive)
    assert np.array_equal(host(d), want)
    assert int(host(total)[0]) == want_total


SIZES = [1, 2, 3, 1023, 1024, 1025, 3 * 1024 + 7, 100003, (1 << 20) - 1, 1 << 20, (1 << 20) + 1, (1 << 21) - 1,
         1 << 21, (1 << 21) + 4097, 3_000_001]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("inclusive", [False, True])
@pytest.mark.parametrize("n", SIZES)
def test_parity(u, op, inclusive, n):
    check(u, values(op, n, 2), op, inclusive)


@pytest.mark.parametrize("n", [5, 100003, (1 << 20) + 3, (1 << 21) + 77])
@pytest.mark.parametrize("op", ["add", "max"])
def test_row_8_bytes_past_16_byte_boundary(u, n, op):
    check(u, values(op, n, 3), op, False, offset=1)
    check(u, values(op, n, 3), op, True, offset=1)


def test_sums_pass_2_64(u):
    n = (1 << 21) + 1000
    a = np.arange(n, dtype=np.uint64) << np.uint64(43)
    check(u, a, "add", False)
    check(u, a, "add", True)


def test_empty_gives_identity(u):
    for op, ident in (("add", 0), ("mul", 1), ("min", (1 << 64) - 1), ("and", (1 << 64) - 1)):
        t = torch.full((1,), 5, dtype=torch.int64, device="cuda")
        u.scan_u64_op(torch.empty(0, dtype=torch.int64, device="cuda"), op, False, t)
        torch.cuda.synchronize()
        assert int(host(t)[0]) == ident


def test_repeated_calls_share_one_workspace(u):
    from u32_prefix_scan_gb300 import _native

    ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_SCAN64, 3_000_001), torch.device("cuda"))
    rng = np.random.default_rng(12)
    for k in range(20):
        n = int(rng.choice([1, 999, 100003, (1 << 21) + 5, 3_000_001]))
        op = OPS[k % len(OPS)]
        check(u, values(op, n, 20 + k), op, bool(k % 2), ws=ws)


@pytest.mark.parametrize("inclusive", [False, True])
def test_full_size(u, inclusive):
    n = 1 << 27
    check(u, inputs.scan_values_u64(n, 2), "add", inclusive)

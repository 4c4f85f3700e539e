"""GPU parity of the scans under every CAIRN integer operator (add, mul,
and, or, xor, min, max) against the CPU oracle, through the C ABI: both
forms, sizes through both launch shapes with ragged tails, misaligned
starts, the identity for n = 0, and the add operator equal to the plain
scan entry points."""

import numpy as np
import pytest

import oracle
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OPS = ["add", "mul", "and", "or", "xor", "min", "max"]
IDENTITY = {"add": 0, "mul": 1, "and": 0xFFFFFFFF, "or": 0, "xor": 0, "min": 0xFFFFFFFF, "max": 0}


@pytest.fixture(scope="module")
def u():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import build

    build.build()
    import u32_prefix_scan_gb300 as u

    return u


def values_for(op, n, seed=3):
    a = inputs.scan_values(n, seed)
    if op == "mul":
        a = a | np.uint32(1)  # odd factors: the wrapped product stays informative
    if op == "and":
        a = a | np.uint32(0xFFFF0FFF)  # mostly ones, so the running and lasts many elements
    if op == "or":
        a = a & np.uint32(0x0000F000) | (a >> np.uint32(31))  # mostly zeros
    return a


def run(u, op, inclusive, a, offset=0):
    buf = torch.empty(a.size + offset + 4, dtype=torch.int32, device="cuda")
    d = buf[offset: offset + a.size]
    d.copy_(torch.from_numpy(a.view(np.int32)))
    total = u.scan_u32_op(d, op, inclusive)
    u.check()
    return d.cpu().numpy().view(np.uint32), int(total.cpu().numpy().view(np.uint32)[0])


SIZES = [1, 2, 33, 2049, 65536 + 3, (1 << 22) + 7, 3 * 16384 * 40 + 11]


@pytest.mark.parametrize("inclusive", [False, True])
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("op", OPS)
def test_operator_scan_parity(u, op, inclusive, n):
    a = values_for(op, n)
    got, total = run(u, op, inclusive, a)
    want, want_total = oracle.scan_op(a, op, inclusive)
    assert np.array_equal(got, want)
    assert total == want_total


@pytest.mark.parametrize("op", ["mul", "min", "xor"])
@pytest.mark.parametrize("offset", [1, 3])
def test_operator_scan_misaligned(u, op, offset):
    n = (1 << 22) + 5
    a = values_for(op, n, 4)
    got, total = run(u, op, True, a, offset)
    want, want_total = oracle.scan_op(a, op, True)
    assert np.array_equal(got, want) and total == want_total


@pytest.mark.parametrize("op", OPS)
def test_empty_gives_identity(u, op):
    total = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    u.scan_u32_op(torch.empty(0, dtype=torch.int32, device="cuda"), op, False, total)
    u.check()
    assert int(total.cpu().numpy().view(np.uint32)[0]) == IDENTITY[op]


def test_add_operator_matches_plain_entry_points(u):
    n = (1 << 22) + 3
    a = inputs.scan_values(n, 8)
    for inclusive in (False, True):
        got, total = run(u, "add", inclusive, a)
        d = torch.from_numpy(a.view(np.int32).copy()).cuda()
        t2 = (u.scan_inclusive_u32 if inclusive else u.scan_exclusive_u32)(d)
        u.check()
        assert np.array_equal(got, d.cpu().numpy().view(np.uint32))
        assert total == int(t2.cpu().numpy().view(np.uint32)[0])


@pytest.mark.parametrize("op", ["max", "mul"])
def test_operator_scan_full_size(u, op):
    n = 1 << 28
    a = values_for(op, n, 2)
    got, total = run(u, op, False, a)
    want, want_total = oracle.scan_op(a, op, False)
    assert np.array_equal(got, want) and total == want_total

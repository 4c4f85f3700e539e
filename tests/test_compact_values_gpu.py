"""GPU parity of the compaction of values (CAIRN's compact ... where ...
yield) against the CPU oracle, through the C ABI: kept values in order at
the front, the rest of `out` untouched, count; flags or the non-zero test;
keep rates 0, 0.1, 0.9 and 1; sizes spanning many tiles with ragged tails;
values and flags at every 4-byte offset mod 16; the page's keep_live
example; repeated calls on one workspace; the full benchmark workload."""

import numpy as np
import pytest

import oracle
from conftest import read_golden
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SENTINEL = 0xA5A5A5A5


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


def flags_for(kind: str, n: int, seed: int = 4) -> np.ndarray:
    if kind in (0.1, 0.9):
        return inputs.compact_flags(n, seed, kind)
    if kind == "none":
        return np.zeros(n, np.int32)
    if kind == "all":
        return np.full(n, -3, np.int32)
    raise ValueError(kind)


def check(u, v, f, off_v=0, off_f=0, off_o=0, ws=None):
    n = v.size
    before = np.full(n, SENTINEL, np.uint32)
    dv = dev(v, off_v)
    df = None if f is None else dev(f, off_f)
    do = dev(before, off_o)
    out, count = u.compact_values_u32(dv, df, do, workspace=ws)
    u.check(workspace=ws)
    want, used = oracle.compact_values(v, f, before)
    assert int(count.item()) == used
    assert np.array_equal(host(out), want)  # front = kept values, rest untouched
    assert np.array_equal(host(dv), v)


SIZES = [1, 2, 7, 8191, 8192, 8193, 14336, 14337, 3 * 14336 + 77, 100003, (1 << 20) + 5]


@pytest.mark.parametrize("kind", [0.1, 0.9, "none", "all"])
@pytest.mark.parametrize("n", SIZES)
def test_with_flags(u, kind, n):
    check(u, inputs.scan_values(n, 4), flags_for(kind, n))


@pytest.mark.parametrize("p", [0.1, 0.9])
@pytest.mark.parametrize("n", SIZES)
def test_nonzero_values(u, p, n):
    v = np.where(inputs.compact_flags(n, 4, p) != 0, inputs.scan_values(n, 4) | np.uint32(1), 0).astype(np.uint32)
    check(u, v, None)


@pytest.mark.parametrize("offs", [(1, 1, 0), (2, 2, 3), (3, 3, 1), (0, 1, 2), (1, 0, 0), (3, 2, 1)])
@pytest.mark.parametrize("n", [9, 3 * 8192 + 5, (1 << 18) + 3])
def test_offsets(u, offs, n):
    v = inputs.scan_values(n, 7)
    check(u, v, flags_for(0.1, n, 7), *offs)
    vz = np.where(flags_for(0.9, n, 7) != 0, v | np.uint32(1), 0).astype(np.uint32)
    check(u, vz, None, offs[0], 0, offs[2])


def test_golden_keep_live(u):
    g = read_golden("cairn_compact_live.txt")
    samples = np.array([int(x) for x in g["samples"].split()], dtype=np.uint32)
    out, count = u.compact_values_u32(dev(samples), None, torch.zeros(samples.size, dtype=torch.int32, device="cuda"))
    u.check()
    assert int(count.item()) == int(g["count"])
    assert host(out).tolist() == [int(x) for x in g["live_after"].split()]


def test_empty(u):
    count = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    u.compact_values_u32(e, None, e, count)
    torch.cuda.synchronize()
    assert int(count.item()) == 0


def test_repeated_calls_share_one_workspace(u):
    from u32_prefix_scan_gb300 import _native

    ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_COMPACT, (1 << 20) + 5), torch.device("cuda"))
    rng = np.random.default_rng(8)
    for k in range(24):
        n = int(rng.choice([1, 777, 8192 * 3, 14336 * 2 + 1, 100003, (1 << 20) + 5]))
        v = inputs.splitmix_u32(11, 0, n, start=k * 1000)
        if k % 2:
            check(u, v, flags_for(0.1 if k % 4 == 1 else 0.9, n, 11 + k), ws=ws)
        else:
            check(u, np.where(v & np.uint32(3), v, 0).astype(np.uint32), None, ws=ws)


@pytest.mark.parametrize("p", [0.1, 0.9])
def test_full_size(u, p):
    n = 1 << 27
    check(u, inputs.scan_values(n, 4), inputs.compact_flags(n, 4, p))

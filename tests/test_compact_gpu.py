"""GPU parity of stream compaction against the CPU oracle, through the C
ABI: bit-exact offsets, indices (kept front, -1 tail) and count for keep
rates from none to all, any non-zero flag value, ragged tails, misaligned
and differently aligned buffers, offsets omitted, repeated calls on one
workspace, and both benchmark workloads at full size (n = 2^27)."""

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


def dev(a: np.ndarray, offset: int = 0, fill: int = 0x5A5A5A5A):
    buf = torch.full((a.size + offset + 4,), fill, dtype=torch.int32, device="cuda")
    view = buf[offset: offset + a.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(a).astype(np.int32)))
    return view


def empty(n: int, offset: int = 0):
    return dev(np.full(n, 0x5A5A5A5A, dtype=np.int32), offset)


def flags_for(kind: str, n: int, seed: int = 4) -> np.ndarray:
    if kind in ("p0.1", "p0.9"):
        return inputs.compact_flags(n, seed, float(kind[1:]))
    if kind == "none":
        return np.zeros(n, np.int32)
    if kind == "all":
        return np.ones(n, np.int32)
    if kind == "mixed":
        f = (inputs.splitmix_u32(seed, 1, n) < np.uint32(1 << 31)).astype(np.int32)
        f[f != 0] = np.where(np.arange(int(f.sum())) % 3 == 0, -7, 123456)  # any non-zero keeps
        return f
    raise ValueError(kind)


def check_compact(u, f, off_f=0, off_o=0, off_i=0, with_offsets=True):
    n = f.size
    fl = dev(f, off_f)
    offsets = empty(n, off_o) if with_offsets else None
    indices = empty(n, off_i)
    _, _, count = u.compact_indices_u32(fl, offsets, indices, want_offsets=with_offsets)
    u.check()
    want_off, want_idx, want_count = oracle.compact_indices(f)
    assert int(count.item()) == want_count
    assert np.array_equal(indices.cpu().numpy(), want_idx)
    if with_offsets:
        assert np.array_equal(offsets.cpu().numpy(), want_off)
    assert np.array_equal(fl.cpu().numpy(), f)  # flags untouched


SIZES = [1, 2, 3, 5, 127, 16384, 16384 + 1, 3 * 16384 + 77, 100003, (1 << 20) + 5]


@pytest.mark.parametrize("kind", ["p0.1", "p0.9", "none", "all", "mixed"])
@pytest.mark.parametrize("n", SIZES)
def test_compact_parity(u, kind, n):
    check_compact(u, flags_for(kind, n))


@pytest.mark.parametrize("offs", [(1, 1, 0), (2, 2, 3), (3, 3, 1), (1, 2, 0), (0, 3, 2), (2, 0, 1)])
@pytest.mark.parametrize("n", [9, 16384 * 3 + 5, (1 << 18) + 3])
def test_compact_misaligned(u, offs, n):
    check_compact(u, flags_for("mixed", n, 5), *offs)


@pytest.mark.parametrize("n", [5, 100003])
def test_compact_without_offsets(u, n):
    check_compact(u, flags_for("p0.1", n), with_offsets=False)


def test_compact_empty(u):
    count = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    u.compact_indices_u32(torch.empty(0, dtype=torch.int32, device="cuda"), count=count)
    u.check()
    assert int(count.item()) == 0


def test_repeated_calls_share_one_workspace(u):
    ws = u.Workspace(1 << 20, torch.device("cuda"))
    rng = np.random.default_rng(6)
    for k in range(24):
        n = int(rng.choice([1, 777, 16384 * 3, 100003, (1 << 20) + 5]))
        f = flags_for(["p0.1", "p0.9", "mixed"][k % 3], n, 10 + k)
        fl = dev(f)
        offsets, indices, count = u.compact_indices_u32(fl, workspace=ws)
        u.check(workspace=ws)
        want_off, want_idx, want_count = oracle.compact_indices(f)
        assert int(count.item()) == want_count, k
        assert np.array_equal(indices.cpu().numpy(), want_idx), k
        assert np.array_equal(offsets.cpu().numpy(), want_off), k


@pytest.mark.parametrize("p", ["p0.1", "p0.9"])
def test_workload_2_27_full_parity(u, p):
    # The compaction benchmark: n = 2^27 int32 flags, Bernoulli(p), seed 4.
    n = 1 << 27
    f = flags_for(p, n)
    check_compact(u, f)

"""GPU parity of the stable radix-sort permutation against the CPU oracle
(and numpy's stable argsort), through the C ABI: uniform keys, tie-heavy
keys, all keys equal, keys differing in one digit only, sorted and reversed
input, ragged tails, repeated calls on one workspace, and both benchmark
workloads at full size (n = 2^25)."""

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


def keys_for(kind: str, n: int, seed: int = 5) -> np.ndarray:
    if kind == "uniform":
        return inputs.radix_keys(n, seed)
    if kind == "ties256":
        return inputs.radix_keys(n, seed, ties=True)
    if kind == "ties65536":
        return inputs.radix_keys(n, seed) >> np.uint32(16)
    if kind == "equal":
        return np.full(n, 0xDEADBEEF, dtype=np.uint32)
    if kind == "top_digit":  # only the most significant digit varies
        return (inputs.radix_keys(n, seed) & np.uint32(0xFF000000)) | np.uint32(0x00ABCDEF)
    if kind == "mid_digit":  # only the second digit varies, set bits on both sides of it
        return (inputs.radix_keys(n, seed) & np.uint32(0x0000FF00)) | np.uint32(0x12340056)
    if kind == "two_values":
        return np.where(inputs.radix_keys(n, seed) & np.uint32(1), np.uint32(7), np.uint32(0xFFFFFFFF))
    if kind == "sorted":
        return np.sort(inputs.radix_keys(n, seed))
    if kind == "reversed":
        return np.sort(inputs.radix_keys(n, seed))[::-1].copy()
    raise ValueError(kind)


def check_perm(u, keys):
    d = torch.from_numpy(keys.view(np.int32).copy()).cuda()
    perm = u.radix_sort_perm_u32(d)
    u.check()
    got = perm.cpu().numpy()
    want = oracle.sort_perm(keys)
    assert np.array_equal(got, want)
    assert np.array_equal(d.cpu().numpy().view(np.uint32), keys)  # keys untouched


# A digit pass takes tiles of 11264 keys (512 threads x 22); sizes around
# one and several tiles, and around 8192 (the tile of the 16-key shape).
TILE = 512 * 22
SIZES = [1, 2, 3, 100, 8191, 8192, 8193, TILE - 1, TILE, TILE + 1, 3 * TILE + 77, 100003, (1 << 20) + 5]


@pytest.mark.parametrize("kind", ["uniform", "ties256", "ties65536", "equal", "top_digit", "mid_digit", "two_values",
                                  "sorted", "reversed"])
@pytest.mark.parametrize("n", SIZES)
def test_radix_parity(u, kind, n):
    check_perm(u, keys_for(kind, n))


def test_radix_agrees_with_numpy_stable_argsort(u):
    keys = keys_for("ties65536", 300007)
    d = torch.from_numpy(keys.view(np.int32).copy()).cuda()
    perm = u.radix_sort_perm_u32(d).cpu().numpy()
    assert np.array_equal(perm, np.argsort(keys, kind="stable").astype(np.int32))


def test_radix_empty(u):
    perm = u.radix_sort_perm_u32(torch.empty(0, dtype=torch.int32, device="cuda"))
    u.check()
    assert perm.numel() == 0


def test_repeated_calls_share_one_workspace(u):
    from u32_prefix_scan_gb300 import _native

    ws = u.Workspace(_native.lib().u32scan_workspace_bytes(_native.OP_RADIX, 100003), torch.device("cuda"))
    rng = np.random.default_rng(8)
    kinds = ["uniform", "ties256", "equal", "top_digit", "two_values"]
    for k in range(15):
        n = int(rng.choice([1, 777, 8192 * 3, 100003]))
        keys = keys_for(kinds[k % len(kinds)], n, 20 + k)
        d = torch.from_numpy(keys.view(np.int32).copy()).cuda()
        perm = u.radix_sort_perm_u32(d, workspace=ws)
        u.check(workspace=ws)
        assert np.array_equal(perm.cpu().numpy(), oracle.sort_perm(keys)), k


@pytest.mark.parametrize("kind", ["uniform", "ties256"])
def test_workload_2_25_full_parity(u, kind):
    # The radix benchmark: n = 2^25 keys u32(5, 0, i), and the [0, 256) variant.
    check_perm(u, keys_for(kind, 1 << 25))


@pytest.mark.parametrize("kind", ["uniform", "ties256", "equal", "top_digit", "mid_digit", "two_values", "reversed"])
@pytest.mark.parametrize("n", [1, 8193, 100003, (1 << 20) + 5])
def test_sort_keys_and_permutation(u, kind, n):
    keys = keys_for(kind, n)
    d = torch.from_numpy(keys.view(np.int32).copy()).cuda()
    out, perm = u.radix_sort_u32(d)
    u.check()
    want_perm = oracle.sort_perm(keys)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), keys[want_perm])  # the oracle's order
    assert np.array_equal(perm.cpu().numpy(), want_perm)
    assert np.array_equal(d.cpu().numpy().view(np.uint32), keys)


@pytest.mark.parametrize("kind", ["uniform", "ties256", "equal", "top_digit", "mid_digit"])
def test_sort_keys_only(u, kind):
    keys = keys_for(kind, 300007)
    d = torch.from_numpy(keys.view(np.int32).copy()).cuda()
    out, perm = u.radix_sort_u32(d, want_perm=False)
    u.check()
    assert perm is None
    assert np.array_equal(out.cpu().numpy().view(np.uint32), keys[oracle.sort_perm(keys)])


@pytest.mark.parametrize("ties", [False, True])
def test_sort_keys_full_size(u, ties):
    keys = inputs.radix_keys(1 << 25, 5, ties=ties)
    d = torch.from_numpy(keys.view(np.int32).copy()).cuda()
    out, perm = u.radix_sort_u32(d)
    u.check()
    want_perm = oracle.sort_perm(keys)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), keys[want_perm])  # the oracle's order
    assert np.array_equal(perm.cpu().numpy(), want_perm)

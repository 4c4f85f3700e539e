"""The allocation-free exclusive scan, through the C ABI.

scan_exclusive_u32_noalloc serves callers that cannot allocate device
memory (and so cannot hand the library a workspace): its carry scratch is a
fixed array inside the library. Its results must equal those of the
allocating entry point, scan_exclusive_u32, bit for bit, on two calls in a
row (the second call finds the first call's leftovers in the shared array),
and the oracle's, element by element, on both launch shapes; a carry wait
that runs out must show in u32scan_check_noalloc and leave later calls
exact.

This file is named to be collected last, so that a failure here stops a
`-x` run only after every other test has run. It must also pass alone in a
fresh process.
"""

import numpy as np
import pytest

import oracle
from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TAG_PERIOD = 1 << 29  # carry-word tags repeat every 2^29 launches


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import _native, build

    build.build()
    return _native.lib()


def _dev(a: np.ndarray):
    return torch.from_numpy(a.view(np.int32).copy()).cuda()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _noalloc(lib, a: np.ndarray):
    """Scan a copy of `a` with the allocation-free entry point; returns the
    scanned array and total on the host and the status word's reading."""
    from u32_prefix_scan_gb300 import _native

    d = _dev(a)
    total = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert lib.scan_exclusive_u32_noalloc(d.data_ptr(), a.size, total.data_ptr(), _stream()) == _native.OK
    status = lib.u32scan_check_noalloc(_stream())
    return d.cpu().numpy().view(np.uint32), int(total.cpu().numpy().view(np.uint32)[0]), status


def test_noalloc_matches_allocating_scan_on_two_calls_in_a_row(lib):
    from u32_prefix_scan_gb300 import _native

    stream = _stream()
    # two different sizes: several wide tiles with a ragged tail, then a
    # smaller array that reuses the scratch the first call left behind
    for call, n in enumerate((3 * (1 << 22) + 12345, 100003)):
        a = inputs.splitmix_u32(21, 0, n, start=call * n)
        ref = _dev(a)
        ref_total = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws_bytes = lib.u32scan_workspace_bytes(_native.OP_SCAN, n)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        assert lib.scan_exclusive_u32(ref.data_ptr(), n, ref_total.data_ptr(), ws.data_ptr(), ws_bytes,
                                      stream) == _native.OK

        got = _dev(a)
        got_total = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        assert lib.scan_exclusive_u32_noalloc(got.data_ptr(), n, got_total.data_ptr(), stream) == _native.OK
        torch.cuda.synchronize()

        assert torch.equal(got, ref), f"call {call}: scanned arrays differ"
        assert torch.equal(got_total, ref_total), f"call {call}: totals differ"


@pytest.mark.parametrize("sizes", [
    # both sides of the 2^19-element switch between the one-tile-per-block
    # kernel (2048-element tiles) and the persistent one (16384)
    ((1 << 19) - 5, (1 << 19) + 77, 1, 2049),
    # a long call, then shorter ones that reuse the front of its carry words
    ((1 << 24) + 12345, 3 * 16384 + 7, 5000, (1 << 19) + 1),
], ids=["crossover", "after-a-larger-call"])
def test_noalloc_matches_the_oracle(lib, sizes):
    from u32_prefix_scan_gb300 import _native

    for k, n in enumerate(sizes):
        a = inputs.splitmix_u32(40 + k, 0, n)
        got, got_total, status = _noalloc(lib, a)
        want, want_total = oracle.scan_exclusive(a)
        assert status == _native.OK, n
        assert np.array_equal(got, want), f"n={n}: scanned array differs from the oracle"
        assert got_total == want_total, f"n={n}: total differs from the oracle"


def test_noalloc_at_its_maximum_size(lib):
    """n = 2^31, the largest size the fixed array serves: all ones gives
    a[j] = j and the total n (the closed form of the exclusive scan)."""
    from u32_prefix_scan_gb300 import _native

    n = 1 << 31
    d = torch.ones(n, dtype=torch.int32, device="cuda")
    total = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.scan_exclusive_u32_noalloc(d.data_ptr(), n, total.data_ptr(), _stream()) == _native.OK
    assert lib.u32scan_check_noalloc(_stream()) == _native.OK
    assert int(total.item()) & 0xffffffff == n
    want = torch.arange(n, dtype=torch.int32, device="cuda")
    assert torch.equal(d, want)
    del d, want
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n,skip", [(2048 * 8, 2), ((1 << 22) + 16384 * 3 + 5, 3)],
                         ids=["one-tile-kernel", "persistent-kernel"])
def test_noalloc_timeout_is_reported_and_later_calls_are_exact(lib, n, skip):
    """A tile that never publishes its carry (test hook) makes the tiles
    after it wait 20 ms, give up and record a timeout in the fixed array's
    status word; u32scan_check_noalloc reports it once and clears it."""
    from u32_prefix_scan_gb300 import _native

    a = inputs.scan_values(n, 11)
    d = _dev(a)
    total = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.u32scan_test_noalloc_skip_publish(d.data_ptr(), n, total.data_ptr(), skip, 20_000_000,
                                                 _stream()) == _native.OK
    assert lib.u32scan_check_noalloc(_stream()) == _native.ETIMEOUT
    assert lib.u32scan_check_noalloc(_stream()) == _native.OK  # cleared
    got, got_total, status = _noalloc(lib, a)
    want, want_total = oracle.scan_exclusive(a)
    assert status == _native.OK
    assert np.array_equal(got, want) and got_total == want_total


def test_noalloc_tag_period_end_clears_old_carry_words(lib):
    """The fixed array's launch count is moved ahead (test hook) so that a
    long call, the launch that ends a tag period, and a long call with the
    long call's tag again follow each other; the third must not take the
    first one's carry words for published ones."""
    from u32_prefix_scan_gb300 import _native

    big = 3 * (1 << 22) + 999
    assert lib.u32scan_test_noalloc_set_epoch(2 * TAG_PERIOD - 2, _stream()) == _native.OK
    for k, n in enumerate((big, 1000)):  # launches 2^30 - 2 and 2^30 - 1 (ends the period)
        a = inputs.splitmix_u32(50 + k, 0, n)
        got, got_total, status = _noalloc(lib, a)
        assert status == _native.OK and np.array_equal(got, oracle.scan_exclusive(a)[0])
    assert lib.u32scan_test_noalloc_set_epoch(3 * TAG_PERIOD - 2, _stream()) == _native.OK  # the long call's tag
    a = inputs.splitmix_u32(52, 0, big)
    got, got_total, status = _noalloc(lib, a)
    want, want_total = oracle.scan_exclusive(a)
    assert status == _native.OK
    assert np.array_equal(got, want) and got_total == want_total, \
        "a carry word from the previous tag period was taken as published"


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    from u32_prefix_scan_gb300 import _native

    fake = 0x10000  # the size check fails first, so nothing is dereferenced
    assert lib.scan_exclusive_u32_noalloc(fake, (1 << 31) + 1, None, None) == _native.EINVAL
    assert lib.u32scan_test_noalloc_skip_publish(fake, (1 << 31) + 1, None, 0, 1000, None) == _native.EINVAL

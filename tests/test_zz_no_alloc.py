"""The allocation-free exclusive scan, through the C ABI.

scan_exclusive_u32_noalloc serves callers that cannot allocate device
memory (and so cannot hand the library a workspace): its carry scratch is a
fixed array inside the library. Its results must equal those of the
allocating entry point, scan_exclusive_u32, bit for bit, on two calls in a
row (the second call finds the first call's leftovers in the shared array).

This file is named to be collected last, so that a failure here stops a
`-x` run only after every other test has run. It must also pass alone in a
fresh process.
"""

import numpy as np
import pytest

from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import _native, build

    build.build()
    return _native.lib()


def _dev(a: np.ndarray):
    return torch.from_numpy(a.view(np.int32).copy()).cuda()


def test_noalloc_matches_allocating_scan_on_two_calls_in_a_row(lib):
    from u32_prefix_scan_gb300 import _native

    stream = torch.cuda.current_stream().cuda_stream
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


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    from u32_prefix_scan_gb300 import _native

    fake = 0x10000  # the size check fails first, so nothing is dereferenced
    assert lib.scan_exclusive_u32_noalloc(fake, (1 << 31) + 1, None, None) == _native.EINVAL

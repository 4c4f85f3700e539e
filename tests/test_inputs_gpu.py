"""The device-side input generator (u32scan_fill_splitmix_u32) against the
host one (inputs.splitmix_u32), bit for bit: counter-based SplitMix64,
u32(seed, stream, i) = high half of mix((seed << 40) | (stream << 32) | i).
Both follow the same published definition; neither is the method's
arithmetic. Also the argument checks."""

import numpy as np
import pytest

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


CASES = [
    (1, 0, 0, 1),
    (2, 0, 0, 1000),
    (3, 1, 0, 1 << 20),
    (5, 0, 12345, (1 << 20) + 7),  # not from index 0
    (4, 1, (1 << 32) - 4099, 4099),  # up to the last index a stream has
    ((1 << 24) - 1, 255, 77, 3001),  # the largest seed and stream
]


@pytest.mark.parametrize("seed,stream,start,n", CASES)
def test_device_draws_equal_host_draws(u, seed, stream, start, n):
    got = u.fill_splitmix_u32(n, seed, stream, start).cpu().numpy().view(np.uint32)
    assert np.array_equal(got, inputs.splitmix_u32(seed, stream, n, start=start))


def test_full_scan_workload_on_the_device(u):
    """The 2^28 scan workload's values, drawn on the device, equal the host's."""
    n = 1 << 28
    d = u.fill_splitmix_u32(n, 2, 0)
    assert np.array_equal(d.cpu().numpy().view(np.uint32), inputs.scan_values(n, 2))


def test_rejected_arguments(u):
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    buf = torch.empty(16, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.u32scan_fill_splitmix_u32(buf.data_ptr(), 0, 1, 0, 0, s) == _native.OK  # nothing to draw
    assert lib.u32scan_fill_splitmix_u32(None, 4, 1, 0, 0, s) == _native.EINVAL
    assert lib.u32scan_fill_splitmix_u32(buf.data_ptr() + 2, 4, 1, 0, 0, s) == _native.EINVAL  # misaligned
    assert lib.u32scan_fill_splitmix_u32(buf.data_ptr(), 4, 1 << 24, 0, 0, s) == _native.EINVAL  # seed too large
    assert lib.u32scan_fill_splitmix_u32(buf.data_ptr(), 4, 1, 256, 0, s) == _native.EINVAL  # stream too large
    assert lib.u32scan_fill_splitmix_u32(buf.data_ptr(), 4, 1, 0, (1 << 32) - 3, s) == _native.EINVAL  # past 2^32
    torch.cuda.synchronize()

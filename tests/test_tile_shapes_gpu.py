"""The same bits from other launch shapes.

"scan.bend source" (header comment) states that the fork depth only sets how
many lanes share the work: every block count gives the same bits. The GPU
counterpart: this library built with other tile shapes (scan tiles of 6
instead of 8 u32x4 a lane, a 3-stage ring, the persistent kernel from 2^17
instead of 2^19 elements; compaction tiles of 6; segmented runs of 3 u32x4
instead of 5 and 5 instead of 7 for the reduce; radix tiles of 8 instead of
16 keys a thread; u64 tiles of 6) must give results identical to the
default library's, bit for bit, on the same seeded inputs: ragged tails,
sizes on both sides of every kernel switch, misaligned starts. Both agree
with the oracle elsewhere; here they are compared with each other.
"""

import numpy as np
import pytest

from u32_prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = ["-DU32SCAN_P_V=6", "-DU32SCAN_P_STAGES=3", "-DU32SCAN_P_MINN_LOG2=17", "-DU32SCAN_C_V=6",
          "-DU32SCAN_CV_V=6", "-DU32SCAN_S_WR4=3", "-DU32SCAN_S_LR=5", "-DU32SCAN_R_KEYS=8", "-DU32SCAN_S64_V=6"]


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from u32_prefix_scan_gb300 import _native, build

    build.build()
    other = _native.load(build.build_variant("shapes", SHAPES))
    return _native.lib(), other


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _ws(lib, op, n):
    b = lib.u32scan_workspace_bytes(op, n)
    return torch.zeros(b, dtype=torch.uint8, device="cuda"), b


def _dev(a, offset=0, dtype=torch.int32):
    """Device copy of a numpy array, `offset` elements into a larger buffer."""
    buf = torch.empty(a.size + offset + 4, dtype=dtype, device="cuda")
    view = buf[offset: offset + a.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int32 if dtype == torch.int32 else np.int64)))
    return view


SIZES = [1, 2047, 2049, 100003, (1 << 17) - 3, (1 << 17) + 5, (1 << 19) + 1, (1 << 22) + 12345]


def _scan(lib, a, inclusive, offset):
    from u32_prefix_scan_gb300 import _native

    d = _dev(a, offset)
    total = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws, wb = _ws(lib, _native.OP_SCAN, a.size)
    fn = lib.scan_inclusive_u32 if inclusive else lib.scan_exclusive_u32
    assert fn(d.data_ptr(), a.size, total.data_ptr(), ws.data_ptr(), wb, _stream()) == _native.OK
    assert lib.u32scan_check(ws.data_ptr(), _stream()) == _native.OK
    return d.clone(), total.clone()


@pytest.mark.parametrize("inclusive", [False, True], ids=["exclusive", "inclusive"])
@pytest.mark.parametrize("n", SIZES)
def test_scan_bits_do_not_depend_on_the_tile_shape(libs, n, inclusive):
    a = inputs.splitmix_u32(71, 0, n)
    for offset in (0, 3):
        x, tx = _scan(libs[0], a, inclusive, offset)
        y, ty = _scan(libs[1], a, inclusive, offset)
        assert torch.equal(x, y) and torch.equal(tx, ty), (n, offset)


@pytest.mark.parametrize("n", [5000, 100003, (1 << 20) + 77, (1 << 22) + 3])
def test_segscan_bits_do_not_depend_on_the_tile_shape(libs, n):
    from u32_prefix_scan_gb300 import _native

    a = inputs.splitmix_u32(72, 0, n)
    f = inputs.segment_heads_geometric(n, 72, log2_mean=6)
    out = []
    for lib in libs:
        for offset in (0, 1):
            d, fl = _dev(a, offset), _dev(f, offset)
            sums = torch.zeros(n, dtype=torch.int32, device="cuda")
            nseg = torch.zeros(1, dtype=torch.int32, device="cuda")
            ws, wb = _ws(lib, _native.OP_SEGSCAN, n)
            assert lib.segscan_inclusive_u32(d.data_ptr(), fl.data_ptr(), n, sums.data_ptr(), n, nseg.data_ptr(),
                                             ws.data_ptr(), wb, _stream()) == _native.OK
            rsums = torch.zeros(n, dtype=torch.int32, device="cuda")
            rn = torch.zeros(1, dtype=torch.int32, device="cuda")
            assert lib.segreduce_u32(_dev(a, offset).data_ptr(), fl.data_ptr(), n, rsums.data_ptr(), n,
                                     rn.data_ptr(), ws.data_ptr(), wb, _stream()) == _native.OK
            assert lib.u32scan_check(ws.data_ptr(), _stream()) == _native.OK
            out.append((d.clone(), sums, nseg, rsums, rn))
    half = len(out) // 2
    for x, y in zip(out[:half], out[half:]):
        assert all(torch.equal(p, q) for p, q in zip(x, y)), n


@pytest.mark.parametrize("n", [777, 100003, (1 << 21) + 5])
def test_compaction_bits_do_not_depend_on_the_tile_shape(libs, n):
    from u32_prefix_scan_gb300 import _native

    f = inputs.compact_flags(n, 73, 0.1)
    v = inputs.splitmix_u32(73, 0, n)
    out = []
    for lib in libs:
        fl = _dev(f, 2)
        off = torch.zeros(n, dtype=torch.int32, device="cuda")
        idx = torch.zeros(n, dtype=torch.int32, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws, wb = _ws(lib, _native.OP_COMPACT, n)
        assert lib.compact_indices_u32(fl.data_ptr(), n, off.data_ptr(), idx.data_ptr(), cnt.data_ptr(),
                                       ws.data_ptr(), wb, _stream()) == _native.OK
        vo = torch.zeros(n, dtype=torch.int32, device="cuda")
        vc = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert lib.compact_values_u32(_dev(v).data_ptr(), fl.data_ptr(), n, vo.data_ptr(), vc.data_ptr(),
                                      ws.data_ptr(), wb, _stream()) == _native.OK
        assert lib.u32scan_check(ws.data_ptr(), _stream()) == _native.OK
        out.append((off, idx, cnt, vo, vc))
    assert all(torch.equal(p, q) for p, q in zip(*out)), n


@pytest.mark.parametrize("ties", [False, True], ids=["uniform", "ties256"])
@pytest.mark.parametrize("n", [1, 4097, 100003, (1 << 21) + 9])
def test_radix_bits_do_not_depend_on_the_tile_shape(libs, n, ties):
    from u32_prefix_scan_gb300 import _native

    keys = inputs.radix_keys(n, 74, ties=ties)
    out = []
    for lib in libs:
        k = _dev(keys, 1)
        perm = torch.zeros(n, dtype=torch.int32, device="cuda")
        ko = torch.zeros(n, dtype=torch.int32, device="cuda")
        ws, wb = _ws(lib, _native.OP_RADIX, n)
        assert lib.radix_sort_u32(k.data_ptr(), n, ko.data_ptr(), perm.data_ptr(), ws.data_ptr(), wb,
                                  _stream()) == _native.OK
        assert lib.u32scan_check(ws.data_ptr(), _stream()) == _native.OK
        out.append((perm, ko))
    assert all(torch.equal(p, q) for p, q in zip(*out)), n


@pytest.mark.parametrize("n", [1000, (1 << 20) + 3, (1 << 21) + 7])
def test_u64_scan_bits_do_not_depend_on_the_tile_shape(libs, n):
    from u32_prefix_scan_gb300 import _native

    a = inputs.scan_values_u64(n, 75)
    out = []
    for lib in libs:
        d = _dev(a, 1, torch.int64)
        total = torch.zeros(1, dtype=torch.int64, device="cuda")
        ws, wb = _ws(lib, _native.OP_SCAN64, n)
        assert lib.scan_u64_op(0, 0, d.data_ptr(), n, total.data_ptr(), ws.data_ptr(), wb, _stream()) == _native.OK
        assert lib.u32scan_check(ws.data_ptr(), _stream()) == _native.OK
        out.append((d.clone(), total))
    assert all(torch.equal(p, q) for p, q in zip(*out)), n

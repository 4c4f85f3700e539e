"""The C ABI without a GPU: the library loads, exports every function that
include/*.h declares, sizes workspaces, and rejects bad arguments on the
host before any CUDA call."""

import ctypes
import pathlib
import re

import pytest

from u32_prefix_scan_gb300 import _native

ROOT = pathlib.Path(__file__).resolve().parents[1]


def declared_functions():
    names = []
    for h in sorted((ROOT / "include").glob("*.h")):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from u32_prefix_scan_gb300 import build

    build.build()
    return _native.lib()


def test_header_declares_the_five_primitives_and_more():
    names = set(declared_functions())
    for must in ("scan_exclusive_u32", "scan_inclusive_u32", "u32scan_workspace_bytes", "u32scan_check"):
        assert must in names


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert name in _native.SIGNATURES, f"{name} has no ctypes signature in the binding"


def test_strerror_and_version(lib):
    for code in (_native.OK, _native.EINVAL, _native.EWORKSPACE, _native.ECUDA, _native.ETIMEOUT):
        assert _native.strerror(code) and _native.strerror(code) != "unknown status"
    assert _native.strerror(12345) == "unknown status"
    assert lib.u32scan_version() >= 100


def test_workspace_bytes(lib):
    wb = lib.u32scan_workspace_bytes
    assert wb(999, 10) == 0
    for n in (0, 1, 1000, 1 << 16, (1 << 22) - 1, 1 << 22, 1 << 28, (1 << 32) - 1):
        b = wb(_native.OP_SCAN, n)
        assert b >= 256 and b % 256 == 0
        # at least one carry word per 16384-element tile (the widest shape)
        assert b >= 256 + 8 * (n // 16384)
    # one 8-byte carry word per tile at most, plus the 256-byte header
    assert wb(_native.OP_SCAN, 1 << 28) <= 256 + 8 * ((1 << 28) // 2048 + 2) + 256


@pytest.mark.parametrize("name", ["scan_exclusive_u32", "scan_inclusive_u32"])
def test_scan_rejects_bad_arguments_on_host(lib, name):
    fn = getattr(lib, name)
    fake = 0x10000  # never dereferenced: every case below fails a host check first
    ws_need = lib.u32scan_workspace_bytes(_native.OP_SCAN, 1000)
    assert fn(None, 10, None, fake, ws_need, None) == _native.EINVAL          # null data
    assert fn(fake + 2, 10, None, fake, ws_need, None) == _native.EINVAL      # misaligned data
    assert fn(fake, 10, fake + 1, fake, ws_need, None) == _native.EINVAL      # misaligned total
    assert fn(fake, 1 << 32, None, fake, 1 << 40, None) == _native.EINVAL     # n too large
    assert fn(fake, 1000, None, None, ws_need, None) == _native.EWORKSPACE    # no workspace
    assert fn(fake, 1000, None, fake, ws_need - 256, None) == _native.EWORKSPACE  # too small
    assert fn(fake, 1000, None, fake + 16, ws_need, None) == _native.EWORKSPACE   # misaligned ws
    # n == 0 with no total: a no-op that touches nothing
    assert fn(None, 0, None, None, 0, None) == _native.OK


def test_radix_workspace_layouts(lib):
    """A radix sort's workspace: small sorts pack their histograms, carry
    words and buffers after the header; from 12 n bytes of buffers at least
    the span other operations' carry words can take (the largest of their
    workspaces for n below 2^32), the carry words come first and everything
    else starts past that span, so a large sort leaves only tagged carry
    words where other operations look."""
    wb = lib.u32scan_workspace_bytes
    reach = max(wb(op, (1 << 32) - 1) for op in (_native.OP_SCAN, _native.OP_SEGSCAN, _native.OP_COMPACT,
                                                  _native.OP_SCAN64))

    def r256(x):
        return -(-x // 256) * 256

    small = 4096 + 256 + 4096 + 256  # histograms, finished-block count, bases, plan
    n0 = -(-reach // 12)  # the first large sort
    for n in (1, 1000, 70001, n0 - 1, n0, (1 << 20) + 5, 1 << 25, 3 << 24):
        carry = r256(8 * 256 * -(-n // 11264))
        bufs = 3 * r256(4 * n)
        if n < n0:
            assert wb(_native.OP_RADIX, n) == 256 + small + carry + bufs, n
        else:
            assert wb(_native.OP_RADIX, n) == max(256 + carry, reach) + small + bufs, n


def test_workspace_init_rejects_null(lib):
    assert lib.u32scan_workspace_init(None, 4096, None) == _native.EWORKSPACE
    assert lib.u32scan_check(None, None) == _native.EWORKSPACE


def test_package_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_native, "SO", tmp_path / "missing.so")
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _native.lib()


@pytest.mark.parametrize("name", ["segscan_inclusive_u32", "segreduce_u32"])
def test_segmented_rejects_bad_arguments_on_host(lib, name):
    fn = getattr(lib, name)
    fake = 0x10000
    need = lib.u32scan_workspace_bytes(_native.OP_SEGSCAN, 1000)
    assert need >= 256 + 16 * (1000 // 8192)
    assert fn(None, fake, 10, fake, 10, fake, fake, need, None) == _native.EINVAL      # null data
    assert fn(fake, None, 10, fake, 10, fake, fake, need, None) == _native.EINVAL      # null flags
    assert fn(fake, fake + 2, 10, fake, 10, fake, fake, need, None) == _native.EINVAL  # misaligned flags
    assert fn(fake, fake, 10, fake + 1, 10, fake, fake, need, None) == _native.EINVAL  # misaligned sums
    assert fn(fake, fake, 1 << 32, fake, 10, fake, fake, 1 << 40, None) == _native.EINVAL
    assert fn(fake, fake, 1000, fake, 10, fake, None, need, None) == _native.EWORKSPACE
    assert fn(fake, fake, 1000, fake, 10, fake, fake, need - 256, None) == _native.EWORKSPACE
    assert fn(None, None, 0, None, 0, None, None, 0, None) == (_native.EINVAL if name == "segreduce_u32"
                                                               else _native.OK)


def test_compact_rejects_bad_arguments_on_host(lib):
    fn = lib.compact_indices_u32
    fake = 0x10000
    need = lib.u32scan_workspace_bytes(_native.OP_COMPACT, 1000)
    assert need >= 256 + 8 * (1000 // 16384)
    assert fn(None, 10, fake, fake, fake, fake, need, None) == _native.EINVAL       # null flags
    assert fn(fake, 10, fake, None, fake, fake, need, None) == _native.EINVAL       # null indices
    assert fn(fake + 1, 10, fake, fake, fake, fake, need, None) == _native.EINVAL   # misaligned flags
    assert fn(fake, 10, fake + 2, fake, fake, fake, need, None) == _native.EINVAL   # misaligned offsets
    assert fn(fake, 1 << 31, fake, fake, fake, fake, 1 << 40, None) == _native.EINVAL  # n too large for int32
    assert fn(fake, 1000, fake, fake, fake, None, need, None) == _native.EWORKSPACE
    assert fn(fake, 1000, fake, fake, fake, fake, need - 256, None) == _native.EWORKSPACE
    assert fn(None, 0, None, None, None, None, 0, None) == _native.OK


def test_radix_rejects_bad_arguments_on_host(lib):
    fn = lib.radix_sort_perm_u32
    fake = 0x10000
    need = lib.u32scan_workspace_bytes(_native.OP_RADIX, 1000)
    assert need >= 3 * 4 * 1000  # two key buffers and one index buffer
    assert fn(None, 10, fake, fake, need, None) == _native.EINVAL
    assert fn(fake, 10, None, fake, need, None) == _native.EINVAL
    assert fn(fake + 2, 10, fake, fake, need, None) == _native.EINVAL
    assert fn(fake, 1 << 31, fake, fake, 1 << 40, None) == _native.EINVAL
    assert fn(fake, 1000, fake, None, need, None) == _native.EWORKSPACE
    assert fn(fake, 1000, fake, fake, need - 256, None) == _native.EWORKSPACE
    assert fn(None, 0, None, None, 0, None) == _native.OK


def test_scan_op_rejects_bad_arguments_on_host(lib):
    fake = 0x10000
    need = lib.u32scan_workspace_bytes(_native.OP_SCAN, 1000)
    for bad_op in (-1, 7, 99):
        assert lib.scan_u32_op(bad_op, 0, fake, 1000, None, fake, need, None) == _native.EINVAL
    assert lib.scan_u32_op(6, 1, None, 10, None, fake, need, None) == _native.EINVAL
    assert lib.scan_u32_op(1, 0, fake, 1000, None, None, need, None) == _native.EWORKSPACE
    assert lib.scan_u32_op(5, 0, None, 0, None, None, 0, None) == _native.OK


def test_radix_sort_rejects_bad_arguments_on_host(lib):
    fn = lib.radix_sort_u32
    fake = 0x100000
    need = lib.u32scan_workspace_bytes(_native.OP_RADIX, 1000)
    assert fn(fake, 10, None, fake, fake, need, None) == _native.EINVAL               # no keys_out
    assert fn(fake, 1000, fake + 400, None, fake, need, None) == _native.EINVAL       # overlapping output
    assert fn(fake, 1000, fake - 400, None, fake, need, None) == _native.EINVAL       # overlapping output
    assert fn(fake, 1000, fake + 4000, fake + 8001, fake, need, None) == _native.EINVAL  # misaligned perm
    assert fn(fake, 1000, fake + 4000, None, None, need, None) == _native.EWORKSPACE
    assert lib.radix_sort_perm_u32(fake, 10, None, fake, need, None) == _native.EINVAL


def test_runs_rejects_bad_arguments_on_host(lib):
    fake = 0x100000
    need = lib.u32scan_workspace_bytes(_native.OP_RUNS, 1000)
    assert need == lib.u32scan_workspace_bytes(_native.OP_SCAN, 1000)
    lay = lib.runs_layout_u32
    assert lay(fake, 1000, None, None, 0, fake, need, None) == _native.EINVAL            # no entries
    assert lay(None, 10, fake, None, 0, fake, need, None) == _native.EINVAL              # no counts
    assert lay(fake, 1000, fake + 400, None, 0, fake, need, None) == _native.EINVAL      # entries inside counts
    assert lay(fake, 1000, fake + 8000, fake + 3996, 8, fake, need, None) == _native.EINVAL  # slots over counts
    assert lay(fake, 1000, fake + 8000, fake + 7996, 8, fake, need, None) == _native.EINVAL  # slots over entries
    assert lay(fake, 1000, fake + 8002, None, 0, fake, need, None) == _native.EINVAL     # misaligned entries
    assert lay(fake, 1 << 31, fake - 8, None, 0, fake, need, None) == _native.EINVAL     # n too large
    assert lay(fake, 1000, fake + 8000, fake + 9000, 1 << 32, fake, need, None) == _native.EINVAL
    assert lay(fake, 1000, fake + 8000, None, 0, None, need, None) == _native.EWORKSPACE
    own = lib.runs_owner_u32
    assert own(None, 10, fake, 4, None) == _native.EINVAL                                # no ends
    assert own(fake, 10, None, 4, None) == _native.EINVAL                                # no owner row
    assert own(fake, 1000, fake + 3996, 4, None) == _native.EINVAL                       # owner over ends
    assert own(fake, 1000, fake + 4002, 4, None) == _native.EINVAL                       # misaligned owner
    assert own(fake, 1 << 31, fake + (1 << 33), 4, None) == _native.EINVAL
    assert own(fake, 10, fake + 4000, 1 << 32, None) == _native.EINVAL
    assert own(fake, 10, None, 0, None) == _native.OK                                    # nothing to write


def test_u8heads_rejects_bad_arguments_on_host(lib):
    fake = 0x100000
    need = lib.u32scan_workspace_bytes(_native.OP_SEGSCAN, 1000)
    for name in ("segscan_inclusive_u32_u8heads", "segreduce_u32_u8heads"):
        fn = getattr(lib, name)
        assert fn(None, fake, 10, fake + 8000, 10, fake + 9000, fake, need, None) == _native.EINVAL
        assert fn(fake, None, 10, fake + 8000, 10, fake + 9000, fake, need, None) == _native.EINVAL
        assert fn(fake + 2, fake, 10, fake + 8000, 10, fake + 9000, fake, need, None) == _native.EINVAL
        assert fn(fake, fake + 4001, 1000, fake + 8000, 10, fake + 9000, None, need, None) == _native.EWORKSPACE
    assert lib.segreduce_u32_u8heads(fake, fake, 10, None, 0, None, fake, need, None) == _native.EINVAL


def test_compact_values_rejects_bad_arguments_on_host(lib):
    fn = lib.compact_values_u32
    fake = 0x100000
    need = lib.u32scan_workspace_bytes(_native.OP_COMPACT, 1000)
    assert fn(None, None, 10, fake, None, fake, need, None) == _native.EINVAL              # no values
    assert fn(fake, None, 10, None, None, fake, need, None) == _native.EINVAL              # no out
    assert fn(fake, None, 1000, fake + 400, None, fake, need, None) == _native.EINVAL      # out over values
    assert fn(fake, fake + 8000, 1000, fake + 9000, None, fake, need, None) == _native.EINVAL  # out over flags
    assert fn(fake + 2, None, 10, fake + 8000, None, fake, need, None) == _native.EINVAL   # misaligned
    assert fn(fake, None, 1 << 31, fake + (1 << 34), None, fake, need, None) == _native.EINVAL
    assert fn(fake, None, 1000, fake + 8000, None, None, need, None) == _native.EWORKSPACE
    assert fn(fake, None, 1000, fake + 8000, None, fake, 256, None) == _native.EWORKSPACE


def test_scan_u64_rejects_bad_arguments_on_host(lib):
    fn = lib.scan_u64_op
    fake = 0x100000
    need = lib.u32scan_workspace_bytes(_native.OP_SCAN64, 1000)
    assert need >= 256 + 16 and need % 256 == 0
    assert fn(7, 0, fake, 1000, None, fake, need, None) == _native.EINVAL        # unknown op
    assert fn(0, 0, None, 10, None, fake, need, None) == _native.EINVAL          # no data
    assert fn(0, 0, fake + 4, 10, None, fake, need, None) == _native.EINVAL      # 4-byte aligned only
    assert fn(0, 1, fake, 10, fake + 12, fake, need, None) == _native.EINVAL     # misaligned total
    assert fn(0, 0, fake, 1 << 32, None, fake, need, None) == _native.EINVAL
    assert fn(0, 0, fake, 1000, None, None, need, None) == _native.EWORKSPACE
    assert fn(0, 0, fake, 1000, None, fake + 8, need, None) == _native.EWORKSPACE  # misaligned workspace


@pytest.mark.parametrize("name", ["scan_exclusive_u32_host", "scan_inclusive_u32_host"])
def test_host_scan_rejects_bad_arguments_on_host(lib, name):
    fn = getattr(lib, name)
    fake = 0x100000  # never dereferenced: every case below fails a check before any CUDA call
    need = lib.u32scan_workspace_bytes(_native.OP_SCAN_HOST, 1000)
    assert fn(None, fake, 10, None, fake, need, None) == _native.EINVAL                 # no input
    assert fn(fake, None, 10, None, fake, need, None) == _native.EINVAL                 # no output
    assert fn(fake + 2, fake + 8000, 10, None, fake, need, None) == _native.EINVAL      # misaligned input
    assert fn(fake, fake + 8001, 10, None, fake, need, None) == _native.EINVAL          # misaligned output
    assert fn(fake, fake + 8000, 10, fake + 9001, fake, need, None) == _native.EINVAL   # misaligned total
    assert fn(fake, fake + 400, 1000, None, fake, need, None) == _native.EINVAL         # partial overlap
    assert fn(fake + 400, fake, 1000, None, fake, need, None) == _native.EINVAL         # partial overlap
    assert fn(fake, fake + 8000, 1 << 62, None, fake, 1 << 40, None) == _native.EINVAL  # n too large


def test_host_scan_workspace_bytes(lib):
    wb = lib.u32scan_workspace_bytes
    for n in (1, 1000, (1 << 18) + 1, 1 << 22, (1 << 25) + 7, 1 << 28, 1 << 34):
        b = wb(_native.OP_SCAN_HOST, n)
        assert b % 256 == 0
        # room for the whole array when it is short, else at least two 2^18-element staging slots
        assert b >= 4 * min(n, 2 << 18)
        # and never more than four 2^23-element slots plus the carry words
        assert b <= 4 * 4 * (1 << 23) + wb(_native.OP_SCAN, 1 << 23) + wb(_native.OP_SCAN, (1 << 22) - 1) + 512


def test_c_example_compiles_and_links(lib, tmp_path):
    # examples/scan_in_place.c built as a caller would build it: the header,
    # the CUDA runtime header, and a link against the library (no GPU call)
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = pathlib.Path("/usr/local/cuda")
    if cc is None or not (cuda / "include" / "cuda_runtime.h").exists():
        pytest.skip("no C compiler or CUDA headers")
    src = ROOT / "examples" / "scan_in_place.c"
    so = pathlib.Path(_native.__file__).with_name("libu32scan.so")
    libdirs = [d for d in (cuda / "lib64", cuda / "targets" / "sbsa-linux" / "lib", cuda / "targets" / "x86_64-linux" / "lib")
               if d.exists()]
    cmd = [cc, "-std=c99", "-Wall", "-Werror", str(src), "-I", str(ROOT / "include"), "-I", str(cuda / "include"),
           str(so), *[f"-L{d}" for d in libdirs], "-lcudart", f"-Wl,-rpath,{so.parent}", "-o", str(tmp_path / "ex")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

"""Every operation keeps the shared 256-byte workspace header (tile counter,
call epoch, device status) valid: interleaving all operations on one
workspace, in every order, must give oracle-exact results and a clean
status after each call."""

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


def dev32(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32).copy()).cuda()


def host_u32(t):
    return t.cpu().numpy().view(np.uint32)


def run_op(u, ws, which, n, seed):
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    if which == "scan":
        a = inputs.splitmix_u32(seed, 0, n)
        d = dev32(a)
        total = u.scan_exclusive_u32(d, workspace=ws)
        want, want_total = oracle.scan_exclusive(a)
        ok = np.array_equal(host_u32(d), want) and int(host_u32(total)[0]) == want_total
    elif which == "segscan":
        a = inputs.splitmix_u32(seed, 0, n)
        f = inputs.segment_heads_geometric(n, seed, log2_mean=6)
        d, fl = dev32(a), dev32(f)
        sums = torch.empty(n, dtype=torch.int32, device="cuda")
        nseg = u.segscan_inclusive_u32(d, fl, sums, workspace=ws)
        want_sums, want_n = oracle.segreduce(a, f)
        ok = (np.array_equal(host_u32(d), oracle.segscan_inclusive(a, f)) and int(nseg.item()) == want_n
              and np.array_equal(host_u32(sums)[:want_n], want_sums))
    elif which == "compact":
        f = inputs.compact_flags(n, seed, 0.1)
        offsets, indices, count = u.compact_indices_u32(dev32(f), workspace=ws)
        wo, wi, wc = oracle.compact_indices(f)
        ok = (np.array_equal(offsets.cpu().numpy(), wo) and np.array_equal(indices.cpu().numpy(), wi)
              and int(count.item()) == wc)
    else:
        k = inputs.radix_keys(n, seed, ties=bool(seed % 2))
        perm = u.radix_sort_perm_u32(dev32(k), workspace=ws)
        ok = np.array_equal(perm.cpu().numpy(), oracle.sort_perm(k))
    status = lib.u32scan_check(ws.ptr, torch.cuda.current_stream().cuda_stream)
    return ok, status


def test_all_operations_share_one_workspace(u):
    from u32_prefix_scan_gb300 import _native

    lib = _native.lib()
    sizes = [1, 5000, 70001, (1 << 22) + 3]
    need = max(lib.u32scan_workspace_bytes(op, n) for op in (1, 2, 3, 4) for n in sizes)
    ws = u.Workspace(need, torch.device("cuda"))
    order = ["scan", "radix", "segscan", "compact", "radix", "scan", "compact", "segscan", "scan", "radix"]
    rng = np.random.default_rng(12)
    for k, which in enumerate(order * 2):
        n = int(rng.choice(sizes))
        ok, status = run_op(u, ws, which, n, 30 + k)
        assert status == _native.OK, (k, which, n)
        assert ok, (k, which, n)

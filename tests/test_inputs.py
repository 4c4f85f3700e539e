"""Pins for the seeded input generator (counter-based SplitMix64)."""

import numpy as np
import pytest

from u32_prefix_scan_gb300 import inputs

MASK64 = (1 << 64) - 1


def splitmix_py(seed, stream, i):
    # Written from Vigna's published SplitMix64 output function, with Python
    # integers (no numpy wraparound semantics involved).
    z = (((seed << 40) | (stream << 32) | i) + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    z ^= z >> 31
    return z >> 32


def test_splitmix_first_output_matches_published_sequence():
    # SplitMix64 started from state 0 first returns 0xE220A8397B1DCDAF; the
    # counter form at seed 0, stream 0, i 0 is that same first output.
    assert splitmix_py(0, 0, 0) == 0xE220A8397B1DCDAF >> 32
    assert int(inputs.splitmix_u32(0, 0, 1)[0]) == 0xE220A839


@pytest.mark.parametrize("seed,stream", [(0, 0), (1, 0), (2, 0), (3, 1), (4, 1), (5, 0), (12345, 7)])
def test_splitmix_matches_python_integers(seed, stream):
    got = inputs.splitmix_u32(seed, stream, 300, start=1000)
    want = [splitmix_py(seed, stream, 1000 + i) for i in range(300)]
    assert got.tolist() == want


def test_threaded_chunks_equal_one_chunk():
    n = (1 << 20) * 3 + 17
    big = inputs.splitmix_u32(2, 0, n)
    pieces = np.concatenate([inputs.splitmix_u32(2, 0, 1 << 20, start=k << 20) for k in range(3)]
                            + [inputs.splitmix_u32(2, 0, 17, start=3 << 20)])
    assert np.array_equal(big, pieces)


def test_workload_shapes_and_rates():
    n = 1 << 20
    small = inputs.scan_values(n, 2, small=True)
    assert small.max() < 16
    heads = inputs.segment_heads_geometric(n, 3)
    assert heads[0] == 1
    assert abs(heads.sum() - n / 1024) < 6 * np.sqrt(n / 1024)
    reg = inputs.segment_heads_regular(n, 4)
    assert reg.sum() == n // 4 and reg[0] == 1 and reg[4] == 1 and reg[1] == 0
    for p in (0.1, 0.9):
        f = inputs.compact_flags(n, 4, p)
        assert abs(f.mean() - p) < 0.005
    ties = inputs.radix_keys(n, 5, ties=True)
    assert ties.max() < 256
    with pytest.raises(ValueError):
        inputs.compact_flags(8, 4, 0.5)
    with pytest.raises(ValueError):
        inputs.splitmix_u32(1, 0, 10, start=(1 << 32) - 5)

"""Seeded synthetic inputs for the U32 scan primitives.

This module is the one piece shared by the CUDA path's tests/benchmark and by
the CPU oracle's tests: it only draws numbers. It holds none of the scan,
segmented-scan, compaction or sort arithmetic, and imports nothing else from
the package.

Generator: counter-based SplitMix64 (S. Vigna's public-domain mixer, the
output function of java.util.SplittableRandom). Element i of stream `stream`
under seed `seed` is

    state = (seed << 40) | (stream << 32) | i          (i < 2^32)
    z = state + 0x9E3779B97F4A7C15                       (mod 2^64)
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9             (mod 2^64)
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB             (mod 2^64)
    z = z ^ (z >> 31)
    u32(seed, stream, i) = z >> 32

Stream 0 draws values/keys, stream 1 draws flags.

Workloads (one per configuration of the benchmark suite):

* scan:        values u32(seed, 0, i); small-value variant u32 >> 28 in [0, 16)
* segmented:   values u32(3, 0, i); heads either Bernoulli(2^-10) from
               u32(3, 1, i) < 2^22 (geometric lengths, mean 1024) with
               index 0 always a head, or every 4th index (length-4 segments)
* compaction:  int32 flags, 1 where u32(4, 1, i) < T, T = round(p * 2^32)
* radix:       keys u32(5, 0, i); tie-heavy variant u32 >> 24 in [0, 256)
* u64 scans:   values u32(seed, 0, 2i) << 32 | u32(seed, 0, 2i + 1), uniform
               over [0, 2^64)
* runs:        per-owner counts from u32(6, 0, i) = d: uniform d >> 29 in
               [0, 8) (mean 3.5, one owner in eight empty), or skewed: d >> 26
               in [0, 64) when d & 15 == 0, else 0 (one owner in sixteen
               holds a run, mean count 1.97)
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "splitmix_u32",
    "scan_values",
    "segment_heads_geometric",
    "segment_heads_regular",
    "compact_flags",
    "radix_keys",
    "run_counts",
    "scan_values_u64",
    "COMPACT_THRESHOLD",
]

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S27, _S30, _S31, _S32 = (np.uint64(k) for k in (27, 30, 31, 32))
_CHUNK = 1 << 20

# Bernoulli thresholds on a u32 draw: flag = draw < T, T = round(p * 2^32).
COMPACT_THRESHOLD = {0.1: 429496730, 0.9: 3865470566}


def _fill(out: np.ndarray, base: np.uint64, start: int, c0: int, c1: int) -> None:
    z = np.arange(start + c0, start + c1, dtype=np.uint64)
    z |= base
    z += _GOLDEN
    z ^= z >> _S30
    z *= _M1
    z ^= z >> _S27
    z *= _M2
    z ^= z >> _S31
    z >>= _S32
    out[c0:c1] = z


def splitmix_u32(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """u32(seed, stream, i) for i in [start, start + n) as a uint32 array."""
    if not (0 <= seed < (1 << 24) and 0 <= stream < 256):
        raise ValueError("seed must be < 2^24 and stream < 256")
    if start < 0 or n < 0 or start + n > (1 << 32):
        raise ValueError("counter range must lie in [0, 2^32)")
    out = np.empty(n, dtype=np.uint32)
    base = np.uint64((seed << 40) | (stream << 32))
    bounds = [(c0, min(n, c0 + _CHUNK)) for c0 in range(0, n, _CHUNK)]
    if len(bounds) <= 2:
        for c0, c1 in bounds:
            _fill(out, base, start, c0, c1)
        return out
    workers = min(len(bounds), os.cpu_count() or 1, 16)
    with ThreadPoolExecutor(max_workers=workers) as pool:
        list(pool.map(lambda b: _fill(out, base, start, b[0], b[1]), bounds))
    return out


def scan_values(n: int, seed: int, small: bool = False) -> np.ndarray:
    """Scan input: uniform u32, or uniform in [0, 16) when `small`."""
    v = splitmix_u32(seed, 0, n)
    if small:
        v >>= np.uint32(28)
    return v


def segment_heads_geometric(n: int, seed: int, log2_mean: int = 10, start: int = 0) -> np.ndarray:
    """int32 head flags, Bernoulli(2^-log2_mean); index 0 always a head.
    Elements start .. start + n - 1 of that array (index 0 only when start
    is 0)."""
    draw = splitmix_u32(seed, 1, n, start=start)
    flags = (draw < np.uint32(1 << (32 - log2_mean))).astype(np.int32)
    if n and start == 0:
        flags[0] = 1
    return flags


def segment_heads_regular(n: int, length: int) -> np.ndarray:
    """int32 head flags: a head every `length` indices, starting at 0."""
    flags = np.zeros(n, dtype=np.int32)
    flags[::length] = 1
    return flags


def compact_flags(n: int, seed: int, p: float, start: int = 0) -> np.ndarray:
    """int32 flags, 1 with probability p (p in COMPACT_THRESHOLD), else 0;
    elements start .. start + n - 1 of the stream."""
    if p not in COMPACT_THRESHOLD:
        raise ValueError(f"p must be one of {sorted(COMPACT_THRESHOLD)}")
    draw = splitmix_u32(seed, 1, n, start=start)
    return (draw < np.uint32(COMPACT_THRESHOLD[p])).astype(np.int32)


def radix_keys(n: int, seed: int, ties: bool = False) -> np.ndarray:
    """Sort keys: uniform u32, or uniform in [0, 256) when `ties`."""
    k = splitmix_u32(seed, 0, n)
    if ties:
        k >>= np.uint32(24)
    return k


def run_counts(n: int, seed: int, skewed: bool = False) -> np.ndarray:
    """uint32 per-owner entry counts: uniform in [0, 8), or (skewed) mostly
    empty with one owner in sixteen holding up to 63 entries."""
    d = splitmix_u32(seed, 0, n)
    if not skewed:
        return d >> np.uint32(29)
    return np.where((d & np.uint32(15)) == 0, d >> np.uint32(26), np.uint32(0)).astype(np.uint32)


def scan_values_u64(n: int, seed: int) -> np.ndarray:
    """uint64 scan input: two consecutive u32 draws per element (high, low)."""
    d = splitmix_u32(seed, 0, 2 * n).astype(np.uint64)
    return (d[0::2] << np.uint64(32)) | d[1::2]

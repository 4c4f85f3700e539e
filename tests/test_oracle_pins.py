"""Pins for the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own loop: each check comes from a value
the pages print (tests/golden/), a closed form, an invariant the pages
state, an independent library routine (numpy), or brute force over every
case of a tiny input.
"""

import itertools

import numpy as np
import pytest

from conftest import read_golden
from u32_prefix_scan_gb300 import inputs

M32 = 1 << 32


# ----------------------------------------------------------------- scan ----

def test_golden_cairn_offsets(oracle_mod):
    g = read_golden("cairn_scan_offsets.txt")
    a = [int(x) for x in g["input"].split()]
    out, total = oracle_mod.scan_exclusive(a)
    for pair in g["expect_at"].split():
        j, v = pair.split(":")
        assert int(out[int(j)]) == int(v)
    assert total == int(g["total"])
    _, total_inc = oracle_mod.scan_inclusive(a)
    assert total_inc == int(g["total"])


@pytest.mark.parametrize("name", ["cairn_reduce_weights.txt", "cairn_tasks_sum.txt"])
def test_golden_cairn_totals(oracle_mod, name):
    g = read_golden(name)
    i = np.arange(int(g["n"]), dtype=np.int64)
    a = {"i%7": i % 7, "i": i}[g["input_formula"]]
    for f in (oracle_mod.scan_exclusive, oracle_mod.scan_inclusive):
        assert f(a)[1] == int(g["total"])


@pytest.mark.parametrize("n", [0, 1, 2, 3, 1000, 100003])
def test_all_ones_closed_form(oracle_mod, n):
    a = np.ones(n, dtype=np.uint32)
    ex, tex = oracle_mod.scan_exclusive(a)
    inc, tinc = oracle_mod.scan_inclusive(a)
    j = np.arange(n, dtype=np.uint64)
    assert np.array_equal(ex, j.astype(np.uint32))
    assert np.array_equal(inc, (j + 1).astype(np.uint32))
    assert tex == tinc == n


def test_iota_triangular_mod_2_32(oracle_mod):
    # a[i] = i: exclusive j(j-1)/2, inclusive j(j+1)/2, both mod 2^32. At
    # n = 2^17 + 5 the triangular numbers pass 2^33, so the wrap is exercised.
    n = (1 << 17) + 5
    a = np.arange(n, dtype=np.uint32)
    j = np.arange(n, dtype=object)
    ex, tex = oracle_mod.scan_exclusive(a)
    inc, tinc = oracle_mod.scan_inclusive(a)
    want_ex = np.array([(x * (x - 1) // 2) % M32 for x in j], dtype=np.uint64)
    want_in = np.array([(x * (x + 1) // 2) % M32 for x in j], dtype=np.uint64)
    assert want_in.max() > 0 and (n * (n - 1) // 2) > 2 * M32
    assert np.array_equal(ex.astype(np.uint64), want_ex)
    assert np.array_equal(inc.astype(np.uint64), want_in)
    assert tex == tinc == (n * (n - 1) // 2) % M32


@pytest.mark.parametrize("seed,n", [(1, 1 << 16), (2, 300001)])
def test_inclusive_is_exclusive_plus_input_and_total(oracle_mod, seed, n):
    a = inputs.scan_values(n, seed)
    ex, tex = oracle_mod.scan_exclusive(a)
    inc, tinc = oracle_mod.scan_inclusive(a)
    assert np.array_equal(inc, ex + a)  # uint32 arithmetic wraps
    wrapped = int(a.astype(np.uint64).sum() % M32)
    assert tex == tinc == wrapped == int(inc[-1])
    # an independent library routine: numpy's wrapping uint32 cumsum
    assert np.array_equal(inc, np.cumsum(a, dtype=np.uint32))


def test_small_values_total_is_exact_sum(oracle_mod):
    # values in [0, 16): the total is below 2^32 even at 2^28 elements, so
    # the wrapped total equals the exact integer sum.
    a = inputs.scan_values(1 << 22, 2, small=True)
    _, t = oracle_mod.scan_exclusive(a)
    assert t == int(a.astype(np.uint64).sum())


def test_brute_force_definition(oracle_mod):
    rng = np.random.default_rng(0)
    for n in range(0, 41):
        a = rng.integers(0, M32, size=n, dtype=np.uint64)
        ex, tex = oracle_mod.scan_exclusive(a)
        inc, tinc = oracle_mod.scan_inclusive(a)
        for j in range(n):
            assert int(ex[j]) == int(sum(int(x) for x in a[:j]) % M32)
            assert int(inc[j]) == int(sum(int(x) for x in a[: j + 1]) % M32)
        assert tex == tinc == int(sum(int(x) for x in a) % M32)


@pytest.mark.parametrize("n", [1, 7, 64, 1000, 4099, 65536, 100003])
def test_every_fork_depth_gives_the_same_bits(oracle_mod, n):
    # scan.bend header: "Every b gives the same bits".
    a = inputs.scan_values(n, 1)
    for inclusive in (False, True):
        plain = (oracle_mod.scan_inclusive if inclusive else oracle_mod.scan_exclusive)(a)
        for b in range(0, 18):
            out, total = oracle_mod.scan_blocked(a, b, inclusive)
            assert np.array_equal(out, plain[0]), (n, b, inclusive)
            assert total == plain[1]


# ------------------------------------------------------------ segmented ----

def _seg_reference_numpy(a, flags):
    """Prefix-difference form with numpy routines: out[j] = C[j] - C[h-1],
    h the last head at or before j (index 0 always a head)."""
    n = a.size
    c = np.cumsum(a, dtype=np.uint32)
    heads = flags != 0
    if n:
        heads[0] = True
    idx = np.where(heads, np.arange(n), 0)
    h = np.maximum.accumulate(idx)
    before = np.where(h > 0, c[np.maximum(h - 1, 0)], np.uint32(0)).astype(np.uint32)
    return c - before


def test_segscan_single_head_is_plain_scan(oracle_mod):
    a = inputs.scan_values(50001, 3)
    flags = np.zeros(a.size, np.int32)
    for f0 in (0, 1):
        flags[0] = f0
        assert np.array_equal(oracle_mod.segscan_inclusive(a, flags), np.cumsum(a, dtype=np.uint32))


def test_segscan_all_heads_is_identity(oracle_mod):
    a = inputs.scan_values(4097, 3)
    assert np.array_equal(oracle_mod.segscan_inclusive(a, np.ones(a.size, np.int32)), a)


@pytest.mark.parametrize("length", [1, 2, 4, 5, 1024])
def test_segscan_regular_segments(oracle_mod, length):
    n = length * 997
    flags = inputs.segment_heads_regular(n, length)
    ones = oracle_mod.segscan_inclusive(np.ones(n, np.uint32), flags)
    assert np.array_equal(ones, (np.arange(n) % length + 1).astype(np.uint32))
    a = inputs.scan_values(n, 3)
    want = np.cumsum(a.reshape(-1, length), axis=1, dtype=np.uint32).reshape(-1)
    assert np.array_equal(oracle_mod.segscan_inclusive(a, flags), want)


def test_segscan_geometric_heads_against_prefix_difference(oracle_mod):
    n = 200003
    a = inputs.scan_values(n, 3)
    flags = inputs.segment_heads_geometric(n, 3)
    flags[flags != 0] = np.where(np.arange(int(flags.sum())) % 2, 1, -9)  # any non-zero is a head
    assert np.array_equal(oracle_mod.segscan_inclusive(a, flags), _seg_reference_numpy(a, flags))


def test_segscan_brute_force_every_head_pattern(oracle_mod):
    n = 9
    a = np.array([5, M32 - 1, 7, 2**31, 3, 2**31 + 1, 11, 1, M32 - 3], dtype=np.uint64)
    for pattern in itertools.product((0, 1), repeat=n):
        flags = np.array(pattern, np.int32)
        out = oracle_mod.segscan_inclusive(a, flags)
        sums, nseg = oracle_mod.segreduce(a, flags)
        want, want_sums = [], []
        for j in range(n):
            h = max([k for k in range(j + 1) if k == 0 or pattern[k]])
            want.append(sum(int(x) for x in a[h : j + 1]) % M32)
        starts = [k for k in range(n) if k == 0 or pattern[k]]
        for s, e in zip(starts, starts[1:] + [n]):
            want_sums.append(sum(int(x) for x in a[s:e]) % M32)
        assert out.tolist() == want, pattern
        assert nseg == len(starts) and sums.tolist() == want_sums, pattern


@pytest.mark.parametrize("kind", ["geometric", "regular4"])
def test_segreduce_invariants(oracle_mod, kind):
    n = 300000
    a = inputs.scan_values(n, 3)
    flags = (inputs.segment_heads_geometric(n, 3) if kind == "geometric"
             else inputs.segment_heads_regular(n, 4))
    sums, nseg = oracle_mod.segreduce(a, flags)
    starts = np.flatnonzero(flags)
    assert nseg == starts.size
    # independent library routine: numpy reduceat over the segment starts
    want = (np.add.reduceat(a.astype(np.uint64), starts) % M32).astype(np.uint32)
    assert np.array_equal(sums, want)
    # segment k's sum is the segmented scan at its last element
    scan = oracle_mod.segscan_inclusive(a, flags)
    ends = np.append(starts[1:], n) - 1
    assert np.array_equal(sums, scan[ends])
    assert int(sums.astype(np.uint64).sum() % M32) == int(a.astype(np.uint64).sum() % M32)


def test_segreduce_empty(oracle_mod):
    sums, nseg = oracle_mod.segreduce(np.zeros(0, np.uint32), np.zeros(0, np.int32))
    assert nseg == 0 and sums.size == 0


# ----------------------------------------------------------- compaction ----

def test_golden_cairn_compact(oracle_mod):
    g = read_golden("cairn_compact_live.txt")
    samples = np.array([int(x) for x in g["samples"].split()])
    offsets, indices, count = oracle_mod.compact_indices((samples > 0).astype(np.int32))
    assert count == int(g["count"])
    assert samples[indices[:count]].tolist() == [int(x) for x in g["front_values"].split()]
    assert indices[count:].tolist() == [-1] * (samples.size - count)
    assert offsets.tolist() == [0, 1, 1, 2]
    live, used = oracle_mod.compact_values(samples)  # `where xs[i] > 0 yield xs[i]` into a zeroed row
    assert used == int(g["count"]) and live.tolist() == [int(x) for x in g["live_after"].split()]


@pytest.mark.parametrize("p", [0.1, 0.9])
def test_compact_against_numpy(oracle_mod, p):
    n = 250007
    flags = inputs.compact_flags(n, 4, p)
    flags[flags != 0] = np.where(np.arange(int(flags.sum())) % 3 == 0, -7, 1)  # any non-zero keeps
    offsets, indices, count = oracle_mod.compact_indices(flags)
    keep = flags != 0
    assert count == int(np.count_nonzero(flags))
    assert np.array_equal(offsets, np.cumsum(keep, dtype=np.int64).astype(np.int32))
    assert np.array_equal(indices[:count], np.flatnonzero(keep).astype(np.int32))
    assert np.all(indices[count:] == -1)
    assert offsets[-1] == count
    assert np.array_equal(np.diff(offsets, prepend=0), keep.astype(np.int32))


def test_compact_degenerate(oracle_mod):
    for n in (0, 1, 5, 1000):
        z = oracle_mod.compact_indices(np.zeros(n, np.int32))
        assert z[2] == 0 and np.all(z[1] == -1) and np.all(z[0] == 0)
        o = oracle_mod.compact_indices(np.ones(n, np.int32))
        assert o[2] == n and np.array_equal(o[1], np.arange(n, dtype=np.int32))


def test_compact_brute_force_every_flag_pattern(oracle_mod):
    n = 10
    for pattern in itertools.product((0, 3), repeat=n):
        flags = np.array(pattern, np.int32)
        offsets, indices, count = oracle_mod.compact_indices(flags)
        kept = [i for i in range(n) if pattern[i]]
        assert count == len(kept)
        assert indices.tolist() == kept + [-1] * (n - len(kept))
        assert offsets.tolist() == [sum(1 for k in range(i + 1) if pattern[k]) for i in range(n)]


# ---------------------------------------------------------------- radix ----

@pytest.mark.parametrize("ties", [False, True])
def test_sort_perm_against_numpy_stable_argsort(oracle_mod, ties):
    keys = inputs.radix_keys(200003, 5, ties=ties)
    want = np.argsort(keys, kind="stable").astype(np.int32)
    assert np.array_equal(oracle_mod.sort_perm(keys), want)


@pytest.mark.parametrize("ties", [False, True])
def test_per_bit_lsd_equals_stable_sort(oracle_mod, ties):
    keys = inputs.radix_keys(30011, 5, ties=ties)
    want = np.argsort(keys, kind="stable").astype(np.int32)
    assert np.array_equal(oracle_mod.radix_perm_bits(keys, 32), want)
    if ties:
        assert np.array_equal(oracle_mod.radix_perm_bits(keys, 8), want)


def test_radix_brute_force_tiny(oracle_mod):
    rng = np.random.default_rng(1)
    for n in range(0, 7):
        for _ in range(25):
            keys = rng.integers(0, 3, size=n).astype(np.uint32)
            keys[rng.random(n) < 0.3] = M32 - 1  # the top bit set too
            good = [p for p in itertools.permutations(range(n))
                    if all((keys[p[i]], p[i]) < (keys[p[i + 1]], p[i + 1]) for i in range(n - 1))]
            assert len(good) == 1  # the stable sorting permutation is unique
            assert oracle_mod.sort_perm(keys).tolist() == list(good[0])
            assert oracle_mod.radix_perm_bits(keys, 32).tolist() == list(good[0])


def test_radix_properties(oracle_mod):
    keys = inputs.radix_keys(100000, 5, ties=True)
    perm = oracle_mod.sort_perm(keys)
    assert np.array_equal(np.sort(perm), np.arange(keys.size, dtype=np.int32))
    s = keys[perm]
    assert np.all(s[1:] >= s[:-1])
    same = s[1:] == s[:-1]
    assert np.all(perm[1:][same] > perm[:-1][same])


# ------------------------------------------------------- operator scans ----

NP_ACCUM = {"add": np.add, "mul": np.multiply, "and": np.bitwise_and, "or": np.bitwise_or,
            "xor": np.bitwise_xor, "min": np.minimum, "max": np.maximum}
IDENTITY = {"add": 0, "mul": 1, "and": M32 - 1, "or": 0, "xor": 0, "min": M32 - 1, "max": 0}


def test_golden_cairn_scan_max(oracle_mod):
    g = read_golden("cairn_scan_max.txt")
    a = [int(x) for x in g["input"].split()]
    out, _ = oracle_mod.scan_op(a, "max", inclusive=True)
    for pair in g["expect_at"].split():
        j, v = pair.split(":")
        assert int(out[int(j)]) == int(v)


def test_golden_cairn_reduce_max(oracle_mod):
    g = read_golden("cairn_reduce_max.txt")
    a = np.arange(int(g["n"])) % 7
    for inclusive in (False, True):
        assert oracle_mod.scan_op(a, "max", inclusive)[1] == int(g["total"])


@pytest.mark.parametrize("op", sorted(NP_ACCUM))
def test_operator_scans_against_numpy_accumulate(oracle_mod, op):
    a = inputs.scan_values(100003, 1)
    if op == "mul":
        a = a | np.uint32(1)  # odd factors keep the wrapped product from collapsing to 0
    want_inc = NP_ACCUM[op].accumulate(a, dtype=np.uint32)
    want_ex = np.concatenate([[np.uint32(IDENTITY[op])], want_inc[:-1]]).astype(np.uint32)
    inc, tinc = oracle_mod.scan_op(a, op, True)
    ex, tex = oracle_mod.scan_op(a, op, False)
    assert np.array_equal(inc, want_inc) and np.array_equal(ex, want_ex)
    assert tinc == tex == int(want_inc[-1])
    e, te = oracle_mod.scan_op(np.zeros(0, np.uint32), op, False)
    assert e.size == 0 and te == IDENTITY[op]


def test_add_operator_is_the_plain_scan(oracle_mod):
    a = inputs.scan_values(5000, 2)
    assert np.array_equal(oracle_mod.scan_op(a, "add", False)[0], oracle_mod.scan_exclusive(a)[0])
    assert np.array_equal(oracle_mod.scan_op(a, "add", True)[0], oracle_mod.scan_inclusive(a)[0])


def test_operator_scans_brute_force(oracle_mod):
    import functools
    import operator

    fns = {"add": lambda x, y: (x + y) % M32, "mul": lambda x, y: (x * y) % M32, "and": operator.and_,
           "or": operator.or_, "xor": operator.xor, "min": min, "max": max}
    rng = np.random.default_rng(5)
    for op, f in fns.items():
        for n in range(0, 12):
            a = [int(x) for x in rng.integers(0, M32, size=n, dtype=np.uint64)]
            inc, _ = oracle_mod.scan_op(a, op, True)
            ex, _ = oracle_mod.scan_op(a, op, False)
            for j in range(n):
                assert int(inc[j]) == functools.reduce(f, a[: j + 1], IDENTITY[op])
                assert int(ex[j]) == functools.reduce(f, a[:j], IDENTITY[op])


# ----------------------------------------------------------------- runs ----

@pytest.mark.parametrize("c", [1, 3, 8])
def test_runs_equal_counts_closed_form(oracle_mod, c):
    n = 1000
    ends, entries, owner = oracle_mod.runs_owner(np.full(n, c, dtype=np.uint32))
    assert np.array_equal(ends, c * np.arange(1, n + 1, dtype=np.uint32))
    assert entries == c * n
    assert np.array_equal(owner, np.arange(c * n, dtype=np.int32) // c)


@pytest.mark.parametrize("skewed", [False, True])
def test_runs_against_numpy(oracle_mod, skewed):
    counts = inputs.run_counts(100003, 6, skewed=skewed)
    ends, entries, owner = oracle_mod.runs_owner(counts)
    want_ends = np.cumsum(counts, dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(ends, want_ends)
    total = int(want_ends[-1])
    assert entries == max(total, 1)
    e = np.arange(total, dtype=np.int64)
    assert np.array_equal(owner, np.searchsorted(want_ends, e, side="right").astype(np.int32))
    # every entry lies inside its owner's run, and no owner is empty
    assert np.all(want_ends[owner] - counts[owner] <= e) and np.all(e < want_ends[owner])


def test_runs_degenerate(oracle_mod):
    for counts in ([], [0], [0, 0, 0]):
        ends, entries, owner = oracle_mod.runs_owner(np.array(counts, dtype=np.uint32))
        assert entries == 1 and owner.tolist() == [-1] and ends.tolist() == [0] * len(counts)
    assert oracle_mod.runs_owner([5])[2].tolist() == [0] * 5
    assert oracle_mod.runs_owner([0, 0, 2, 0, 1, 0])[2].tolist() == [2, 2, 4]
    ends, _ = oracle_mod.runs_layout([M32 - 1, 1])  # ends wrap like the scan
    assert ends.tolist() == [M32 - 1, 0]


def test_runs_brute_force(oracle_mod):
    for n in range(0, 5):
        for counts in itertools.product(range(3), repeat=n):
            ends, entries, owner = oracle_mod.runs_owner(list(counts))
            walk = [i for i, c in enumerate(counts) for _ in range(c)]
            assert owner.tolist() == (walk or [-1])
            assert entries == max(len(walk), 1)
            assert ends.tolist() == [sum(counts[: i + 1]) for i in range(n)]


# ------------------------------------------------------ compact values ----

@pytest.mark.parametrize("p", [0.1, 0.9])
def test_compact_values_against_numpy(oracle_mod, p):
    n = 100003
    v = inputs.scan_values(n, 4)
    f = inputs.compact_flags(n, 4, p)
    before = inputs.scan_values(n, 9)
    out, used = oracle_mod.compact_values(v, f, before)
    keep = v[f != 0]
    assert used == keep.size == np.count_nonzero(f)
    assert np.array_equal(out[:used], keep)
    assert np.array_equal(out[used:], before[used:])  # the rest of out is unchanged


def test_compact_values_nonzero_test(oracle_mod):
    v = np.where(inputs.compact_flags(5000, 4, 0.1) != 0, inputs.scan_values(5000, 4), 0).astype(np.uint32)
    out, used = oracle_mod.compact_values(v)
    assert used == np.count_nonzero(v) and np.array_equal(out[:used], v[v != 0]) and not out[used:].any()
    # flags decide alone: a kept zero value and a dropped non-zero value
    out, used = oracle_mod.compact_values([0, 5, 6], [1, 0, -2], [9, 9, 9])
    assert used == 2 and out.tolist() == [0, 6, 9]


def test_compact_values_brute_force(oracle_mod):
    for n in range(0, 7):
        for bits in range(1 << n):
            f = [(bits >> i) & 1 for i in range(n)]
            v = [10 + i for i in range(n)]
            out, used = oracle_mod.compact_values(v, f, [99] * n)
            kept = [v[i] for i in range(n) if f[i]]
            assert used == len(kept) and out.tolist() == kept + [99] * (n - len(kept))


# ------------------------------------------------------------ u64 scans ----

M64 = 1 << 64
IDENTITY64 = {"add": 0, "mul": 1, "and": M64 - 1, "or": 0, "xor": 0, "min": M64 - 1, "max": 0}


@pytest.mark.parametrize("op", sorted(NP_ACCUM))
def test_u64_operator_scans_against_numpy_accumulate(oracle_mod, op):
    a = inputs.scan_values_u64(50003, 1)
    if op == "mul":
        a = a | np.uint64(1)
    want_inc = NP_ACCUM[op].accumulate(a, dtype=np.uint64)
    want_ex = np.concatenate([[np.uint64(IDENTITY64[op])], want_inc[:-1]]).astype(np.uint64)
    inc, tinc = oracle_mod.scan_op_u64(a, op, True)
    ex, tex = oracle_mod.scan_op_u64(a, op, False)
    assert np.array_equal(inc, want_inc) and np.array_equal(ex, want_ex)
    assert tinc == tex == int(want_inc[-1])
    e, te = oracle_mod.scan_op_u64(np.zeros(0, np.uint64), op, False)
    assert e.size == 0 and te == IDENTITY64[op]


def test_u64_add_wraps_at_2_64_not_2_32(oracle_mod):
    # iota times 2^40: the sums pass 2^64 within 2^24 + 1 terms
    n = (1 << 24) + 1000
    a = np.arange(n, dtype=np.uint64) << np.uint64(40)
    out, total = oracle_mod.scan_op_u64(a, "add", False)
    for j in (1, 1 << 12, 1 << 23, (1 << 24) + 999):
        assert int(out[j]) == ((j * (j - 1) // 2) << 40) % M64
    assert total == ((n * (n - 1) // 2) << 40) % M64


def test_u64_brute_force(oracle_mod):
    import functools
    import operator

    fns = {"add": lambda x, y: (x + y) % M64, "mul": lambda x, y: (x * y) % M64, "and": operator.and_,
           "or": operator.or_, "xor": operator.xor, "min": min, "max": max}
    rng = np.random.default_rng(6)
    for op, f in fns.items():
        for n in range(0, 10):
            a = [int(x) for x in rng.integers(0, M64, size=n, dtype=np.uint64)]
            inc, t = oracle_mod.scan_op_u64(a, op, True)
            ex, _ = oracle_mod.scan_op_u64(a, op, False)
            want = [functools.reduce(f, a[: j + 1]) for j in range(n)]
            assert inc.tolist() == want
            assert ex.tolist() == [IDENTITY64[op]] + want[:-1] if n else ex.tolist() == []
            assert t == (want[-1] if n else IDENTITY64[op])

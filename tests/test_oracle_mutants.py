"""The oracle's pins have teeth: plausible mistakes planted in copies of
oracle.c (on the CPU only) must each fail at least one pin.

Each mutant is one textual edit of the C source, compiled into a temporary
library and bound in place of the real one while a handful of pin tests run.
Every planted edit keeps all memory accesses in bounds.
"""

import contextlib
import ctypes
import pathlib
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = pathlib.Path(oracle.__file__).resolve().parent / "oracle.c"

# (name, original text, planted text, pin tests that must catch it)
MUTANTS = [
    ("exclusive_stores_through_j", "a[j] = s;\n        s = s + x;", "s = s + x;\n        a[j] = s;",
     ["all_ones", "iota", "golden_offsets"]),
    ("inclusive_drops_running_sum", "++j) {\n        s = s + a[j];", "++j) {\n        s = a[j];",
     ["all_ones", "iota", "incl_excl"]),
    ("blocked_pass3_drops_base", "uint32_t run = s[i];", "uint32_t run = 0;", ["fork_depth"]),
    ("blocked_pass2_inclusive", "s[i] = total;\n        total = total + x;",
     "total = total + x;\n        s[i] = total;", ["fork_depth"]),
    ("segscan_positive_heads_only", "if (j == 0 || flags[j] != 0)\n            s = 0;",
     "if (j == 0 || flags[j] > 0)\n            s = 0;", ["seg_geometric"]),
    ("segreduce_drops_last_segment", "if (n != 0)\n        seg_sums[nseg - 1] = s;", "",
     ["seg_brute", "segreduce_inv"]),
    ("compact_offsets_exclusive", "run += (flags[i] != 0) ? 1 : 0;\n        offsets[i] = run;",
     "offsets[i] = run;\n        run += (flags[i] != 0) ? 1 : 0;", ["compact_numpy", "compact_brute"]),
    ("compact_counts_raw_flags", "total += (flags[i] != 0) ? 1 : 0;", "total += flags[i] > 0 ? flags[i] : 0;",
     ["compact_numpy"]),
    ("sort_skips_bit0", "for (unsigned bit = 0; bit < bits; ++bit)",
     "for (unsigned bit = 1; bit < bits; ++bit)", ["lsd", "radix_brute"]),
    ("min_identity_zero", "case 2: case 5: return 0xffffffffu;", "case 2: return 0xffffffffu;",
     ["opscan_min"]),
    ("sort_ties_descending", "return (a->idx > b->idx) - (a->idx < b->idx);",
     "return (a->idx < b->idx) - (a->idx > b->idx);", ["sort_numpy", "radix_brute"]),
    ("runs_ends_exclusive", "run += counts[i];\n        ends[i] = run;", "ends[i] = run;\n        run += counts[i];",
     ["runs_closed", "runs_numpy"]),
    ("runs_entries_may_be_zero", "return run > 0 ? run : 1u;", "return run;", ["runs_degenerate"]),
    ("runs_fill_starts_one_late", "(uint64_t)ends[i] - (uint64_t)counts[i];",
     "(uint64_t)ends[i] - (uint64_t)counts[i] + 1;", ["runs_closed", "runs_brute"]),
    ("compact_values_positive_flags_only", "int keep = flags ? flags[i] != 0 : values[i] != 0;",
     "int keep = flags ? flags[i] > 0 : values[i] != 0;", ["cvalues_nonzero"]),
    ("compact_values_projects_index", "out[used++] = values[i];", "out[used++] = (uint32_t)i;",
     ["cvalues_numpy", "golden_compact"]),
    ("u64_add_truncates_to_32_bits", "case 0: return x + y;\n    case 1: return x * y;\n    case 2: return x & y;\n    case 3: return x | y;\n    case 4: return x ^ y;\n    case 5: return x < y ? x : y;\n    default: return x > y ? x : y;\n    }\n}\n\nstatic uint64_t oracle_identity64",
     "case 0: return (uint32_t)(x + y);\n    case 1: return x * y;\n    case 2: return x & y;\n    case 3: return x | y;\n    case 4: return x ^ y;\n    case 5: return x < y ? x : y;\n    default: return x > y ? x : y;\n    }\n}\n\nstatic uint64_t oracle_identity64",
     ["u64_wrap", "u64_numpy_add"]),
]

PINS = {
    "all_ones": lambda o: [pins.test_all_ones_closed_form(o, n) for n in (3, 1000)],
    "iota": lambda o: pins.test_iota_triangular_mod_2_32(o),
    "golden_offsets": lambda o: pins.test_golden_cairn_offsets(o),
    "incl_excl": lambda o: pins.test_inclusive_is_exclusive_plus_input_and_total(o, 1, 1 << 16),
    "fork_depth": lambda o: [pins.test_every_fork_depth_gives_the_same_bits(o, n) for n in (1000, 4099)],
    "seg_geometric": lambda o: pins.test_segscan_geometric_heads_against_prefix_difference(o),
    "seg_brute": lambda o: pins.test_segscan_brute_force_every_head_pattern(o),
    "segreduce_inv": lambda o: pins.test_segreduce_invariants(o, "geometric"),
    "compact_numpy": lambda o: pins.test_compact_against_numpy(o, 0.1),
    "compact_brute": lambda o: pins.test_compact_brute_force_every_flag_pattern(o),
    "lsd": lambda o: pins.test_per_bit_lsd_equals_stable_sort(o, True),
    "radix_brute": lambda o: pins.test_radix_brute_force_tiny(o),
    "sort_numpy": lambda o: pins.test_sort_perm_against_numpy_stable_argsort(o, True),
    "opscan_min": lambda o: pins.test_operator_scans_against_numpy_accumulate(o, "min"),
    "runs_closed": lambda o: pins.test_runs_equal_counts_closed_form(o, 3),
    "runs_numpy": lambda o: pins.test_runs_against_numpy(o, True),
    "runs_degenerate": lambda o: pins.test_runs_degenerate(o),
    "runs_brute": lambda o: pins.test_runs_brute_force(o),
    "cvalues_nonzero": lambda o: pins.test_compact_values_nonzero_test(o),
    "cvalues_numpy": lambda o: pins.test_compact_values_against_numpy(o, 0.1),
    "golden_compact": lambda o: pins.test_golden_cairn_compact(o),
    "u64_wrap": lambda o: pins.test_u64_add_wraps_at_2_64_not_2_32(o),
    "u64_numpy_add": lambda o: pins.test_u64_operator_scans_against_numpy_accumulate(o, "add"),
}


@contextlib.contextmanager
def bound(lib):
    old = oracle._lib
    oracle._lib = lib
    try:
        yield oracle
    finally:
        oracle._lib = old


def test_real_oracle_passes_the_selected_pins(oracle_mod):
    for check in PINS.values():
        check(oracle_mod)


@pytest.mark.parametrize("name,orig,planted,catchers", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, oracle_mod, name, orig, planted, catchers):
    src = SRC.read_text()
    assert src.count(orig) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / f"{name}.c"
    mutated.write_text(src.replace(orig, planted))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(mutated)])
    lib = oracle._configure(ctypes.CDLL(str(so)))
    with bound(lib) as o:
        for c in catchers:
            with pytest.raises(AssertionError):
                PINS[c](o)

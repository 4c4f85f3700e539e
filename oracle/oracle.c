/*
 * oracle.c -- plain, sequential CPU oracle for the U32 scan primitives.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path
 * (the CUDA library and its binding) never calls it, and the two share no
 * code: no headers, helpers, tables or constants.
 *
 * Every function is one thread, one walk over the data, in the order the
 * source pages give, with no blocking or fusion beyond what the pages state.
 * Arithmetic on values is uint32_t, so every sum wraps at 2^32.
 *
 * Sources (page title, then the part of the page):
 *   [scan.bend]  "scan.bend source" (bendlib): header comment ("Sums wrap",
 *                "Three passes"), sections "Loops (one lane)", "Pass 1",
 *                "Pass 3", "Driver", "API".
 *   [CAIRN]      "Concurrency" (CAIRN docs): sections "reduce and compact",
 *                "scan".
 *   [Futhark]    "Futhark.Pass.ExtractKernels.Segmented":
 *                regularSegmentedRedomap, regularSegmentedScan.
 *   [entelechy]  "parallel" package reference (entelechy docs): kernels
 *                compact_blank / compact_offsets / compact_total /
 *                compact_gather, sort_identity / sort_blank / sort_zeros /
 *                sort_place / sort_next_bit, runs_ends / runs_entries /
 *                runs_slots, graphs compact, sort and runs, function owner.
 *   [CAIRN compact] "Concurrency" (CAIRN docs), "reduce and compact": the
 *                `compact out for i in n where p yield e` collector.
 *
 * Readings taken where the pages are silent (all restated in the design
 * notes): any n is scanned in full (not only 2^floor(log2 n) entries);
 * n = 0 gives total 0; index 0 always opens a segment; a head flag or a
 * compaction flag is "set" when non-zero; compaction fills unused index
 * slots with -1; sort keys are unsigned 32-bit and all 32 bits are sorted;
 * run counts are unsigned 32-bit; owner(e, ends) is the owner whose run
 * holds entry e, -1 for the one slot of a layout with no entries.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * Scan.  [scan.bend] "Loops (one lane)": ex.go sets a[j] to the running sum
 * s before j, then adds the old a[j] into s; in.go adds first and stores the
 * sum through j. "API": exclusive/inclusive return the array and the total
 * a[0] + .. + a[n-1]. Header: "Sums wrap at 2^32, as U32.add does".
 * ---------------------------------------------------------------------- */

uint32_t oracle_scan_exclusive_u32(uint32_t *a, uint64_t n)
{
    uint32_t s = 0;
    for (uint64_t j = 0; j < n; ++j) {
        uint32_t x = a[j];
        a[j] = s;
        s = s + x;
    }
    return s;
}

uint32_t oracle_scan_inclusive_u32(uint32_t *a, uint64_t n)
{
    uint32_t s = 0;
    for (uint64_t j = 0; j < n; ++j) {
        s = s + a[j];
        a[j] = s;
    }
    return s;
}

/*
 * [scan.bend] header "Three passes" and "Driver": the same scan, cut into
 * 2^d blocks (d = the fork depth b, lowered to floor(log2 n)).
 *   pass 1 ("Pass 1", sums.leaf): block i's wrapped sum into s[i];
 *   pass 2: s becomes its exclusive scan (the blocks' bases) and the total;
 *   pass 3 ("Pass 3", puts.leaf): block i rescanned in place from base s[i].
 * The page's blocks are 2^e entries over a power-of-two n; here a block is
 * ceil(n / 2^d) entries so that every n is covered (the last blocks may be
 * short or empty). Pass 2 runs on one lane, as the page does below 2^12
 * sums; above that the page recurses, which gives the same bits.
 * `s` is caller scratch of 2^d entries (d <= 30 as clamped here).
 * Used to pin the page's claim that every b gives the same bits.
 */
uint32_t oracle_scan_blocked_u32(int inclusive, unsigned b, uint32_t *a,
                                 uint64_t n, uint32_t *s)
{
    if (n == 0)
        return 0;
    unsigned lg = 0;
    while ((lg + 1) < 64 && (UINT64_C(1) << (lg + 1)) <= n)
        ++lg;
    unsigned d = b < lg ? b : lg;
    if (d > 30)
        d = 30;
    uint64_t blocks = UINT64_C(1) << d;
    uint64_t len = (n + blocks - 1) / blocks;

    /* pass 1 */
    for (uint64_t i = 0; i < blocks; ++i) {
        uint32_t sum = 0;
        for (uint64_t j = i * len; j < (i + 1) * len && j < n; ++j)
            sum = sum + a[j];
        s[i] = sum;
    }
    /* pass 2: exclusive scan of the block sums, one lane */
    uint32_t total = 0;
    for (uint64_t i = 0; i < blocks; ++i) {
        uint32_t x = s[i];
        s[i] = total;
        total = total + x;
    }
    /* pass 3: each block's scan from its base */
    for (uint64_t i = 0; i < blocks; ++i) {
        uint32_t run = s[i];
        for (uint64_t j = i * len; j < (i + 1) * len && j < n; ++j) {
            uint32_t x = a[j];
            if (inclusive) {
                run = run + x;
                a[j] = run;
            } else {
                a[j] = run;
                run = run + x;
            }
        }
    }
    return total;
}

/* ------------------------------------------------------------------------
 * Scans under the other operators of the CAIRN "Concurrency" page, section
 * "reduce and compact" (the operators of reduce, which scan shares per
 * section "scan"): add_wrap, mul_wrap, &, |, ^, min and max on integers,
 * here on uint32. Each is associative and commutative, with identity 0, 1,
 * all ones, 0, 0, all ones and 0. Exclusive: a[j] = e . a[0] . .. . a[j-1]
 * (e the identity); inclusive: through a[j]; returns the fold of all n.
 * op: 0 add, 1 mul, 2 and, 3 or, 4 xor, 5 min, 6 max.
 * ---------------------------------------------------------------------- */

static uint32_t oracle_apply(int op, uint32_t x, uint32_t y)
{
    switch (op) {
    case 0: return x + y;
    case 1: return x * y;
    case 2: return x & y;
    case 3: return x | y;
    case 4: return x ^ y;
    case 5: return x < y ? x : y;
    default: return x > y ? x : y;
    }
}

static uint32_t oracle_identity(int op)
{
    switch (op) {
    case 1: return 1u;
    case 2: case 5: return 0xffffffffu;
    default: return 0u;
    }
}

uint32_t oracle_scan_op_u32(int op, int inclusive, uint32_t *a, uint64_t n)
{
    uint32_t s = oracle_identity(op);
    for (uint64_t j = 0; j < n; ++j) {
        uint32_t x = a[j];
        if (inclusive) {
            s = oracle_apply(op, s, x);
            a[j] = s;
        } else {
            a[j] = s;
            s = oracle_apply(op, s, x);
        }
    }
    return s;
}

/* ------------------------------------------------------------------------
 * Segmented scan and reduce.  [Futhark] regularSegmentedScan names the
 * segmented scan; regularSegmentedRedomap reduces "until there is only a
 * single value per segment". Segments are marked by head flags: a non-zero
 * flag at j starts a new segment at j, and index 0 always starts one.
 * The definition: out[j] = a[h] + .. + a[j], h the last head at or before j.
 * ---------------------------------------------------------------------- */

void oracle_segscan_inclusive_u32(uint32_t *a, const int32_t *flags, uint64_t n)
{
    uint32_t s = 0;
    for (uint64_t j = 0; j < n; ++j) {
        if (j == 0 || flags[j] != 0)
            s = 0;
        s = s + a[j];
        a[j] = s;
    }
}

/* seg_sums gets one wrapped sum per segment, in segment order; returns the
 * number of segments (0 when n = 0). seg_sums must hold that many. */
uint64_t oracle_segreduce_u32(const uint32_t *a, const int32_t *flags,
                              uint64_t n, uint32_t *seg_sums)
{
    uint64_t nseg = 0;
    uint32_t s = 0;
    for (uint64_t j = 0; j < n; ++j) {
        if (j == 0 || flags[j] != 0) {
            if (j != 0)
                seg_sums[nseg - 1] = s;
            ++nseg;
            s = 0;
        }
        s = s + a[j];
    }
    if (n != 0)
        seg_sums[nseg - 1] = s;
    return nseg;
}

/* ------------------------------------------------------------------------
 * Stream compaction.  [entelechy] graph "compact": flags in (non-zero keeps
 * an element); the kept indices gathered to the front; their count out.
 * Its four kernels, in their order:
 *   compact_blank   -- every slot -1 ("what a slot holds when nothing was
 *                      gathered into it");
 *   compact_offsets -- inclusive prefix sum, so a kept i belongs at
 *                      offsets[i] - 1; the summed term is the keep
 *                      indicator (flag != 0);
 *   compact_total   -- how many were kept, as a row of one;
 *   compact_gather  -- each kept index scattered to its rank with max; a
 *                      zero flag addresses -1 and is dropped.
 * [CAIRN] "reduce and compact": the kept elements land in order at the
 * front. Returns the count (also stored to *count).
 * ---------------------------------------------------------------------- */

int32_t oracle_compact_indices(const int32_t *flags, uint64_t n,
                               int32_t *offsets, int32_t *indices,
                               int32_t *count)
{
    /* compact_blank */
    for (uint64_t i = 0; i < n; ++i)
        indices[i] = -1;
    /* compact_offsets */
    int32_t run = 0;
    for (uint64_t i = 0; i < n; ++i) {
        run += (flags[i] != 0) ? 1 : 0;
        offsets[i] = run;
    }
    /* compact_total (a reduce over the flags) */
    int32_t total = 0;
    for (uint64_t i = 0; i < n; ++i)
        total += (flags[i] != 0) ? 1 : 0;
    /* compact_gather */
    for (uint64_t i = 0; i < n; ++i) {
        int64_t slot = (flags[i] != 0) ? (int64_t)offsets[i] - 1 : -1;
        if (slot < 0 || (uint64_t)slot >= n)
            continue; /* an address outside the target is dropped */
        if ((int32_t)i > indices[slot])
            indices[slot] = (int32_t)i;
    }
    *count = total;
    return total;
}

/* ------------------------------------------------------------------------
 * Radix-sort permutation.  [entelechy] graph "sort": the permutation that
 * orders the keys, least significant bit first, one bit per pass:
 *   sort_identity -- every element starts at its own place (order = iota);
 *   per bit:
 *     sort_zeros  -- zeros[i] = how many of keys[order[0..i]] have a zero
 *                    at this bit (inclusive count);
 *     sort_blank  -- the row the pass scatters into (-1);
 *     sort_place  -- a zero at this bit lands at its rank among the zeros,
 *                    zeros[i] - 1; a one lands behind all Z zeros at its
 *                    rank among the ones, Z + i - zeros[i]; scatter with
 *                    max (each place is written exactly once);
 *     sort_next_bit -- on to the next bit.
 * Keys are unsigned 32-bit here and `bits` of them (1..32) are sorted.
 * zeros and slots are caller scratch of n entries each.
 * ---------------------------------------------------------------------- */

void oracle_radix_perm_bits(const uint32_t *keys, uint64_t n, unsigned bits,
                            int32_t *perm, int32_t *zeros, int32_t *slots)
{
    /* sort_identity */
    for (uint64_t i = 0; i < n; ++i)
        perm[i] = (int32_t)i;
    for (unsigned bit = 0; bit < bits; ++bit) {
        /* sort_zeros */
        int32_t z = 0;
        for (uint64_t i = 0; i < n; ++i) {
            z += ((keys[perm[i]] >> bit) & 1u) == 0 ? 1 : 0;
            zeros[i] = z;
        }
        int32_t Z = n ? zeros[n - 1] : 0;
        /* sort_blank */
        for (uint64_t i = 0; i < n; ++i)
            slots[i] = -1;
        /* sort_place */
        for (uint64_t i = 0; i < n; ++i) {
            int64_t place;
            if (((keys[perm[i]] >> bit) & 1u) == 0)
                place = (int64_t)zeros[i] - 1;
            else
                place = (int64_t)Z + (int64_t)i - (int64_t)zeros[i];
            if (perm[i] > slots[place])
                slots[place] = perm[i];
        }
        /* sort_next_bit: the placed row is the next pass's order */
        memcpy(perm, slots, (size_t)n * sizeof(int32_t));
    }
}

/*
 * The same permutation by its definition: the unique stable sorting
 * permutation, i.e. the indices ordered by (key, index). The library sort
 * (qsort) serves as the one step; the comparator is a total order, so the
 * result does not depend on qsort's own stability.
 */
typedef struct {
    uint32_t key;
    int32_t idx;
} oracle_pair;

static int oracle_pair_cmp(const void *pa, const void *pb)
{
    const oracle_pair *a = (const oracle_pair *)pa;
    const oracle_pair *b = (const oracle_pair *)pb;
    if (a->key != b->key)
        return a->key < b->key ? -1 : 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

/* Returns 0, or -1 if the pair buffer cannot be allocated. */
int oracle_sort_perm_u32(const uint32_t *keys, uint64_t n, int32_t *perm)
{
    if (n == 0)
        return 0;
    oracle_pair *p = (oracle_pair *)malloc((size_t)n * sizeof(oracle_pair));
    if (!p)
        return -1;
    for (uint64_t i = 0; i < n; ++i) {
        p[i].key = keys[i];
        p[i].idx = (int32_t)i;
    }
    qsort(p, (size_t)n, sizeof(oracle_pair), oracle_pair_cmp);
    for (uint64_t i = 0; i < n; ++i)
        perm[i] = p[i].idx;
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------
 * Runs.  [entelechy] graph "runs": from each owner's count of entries,
 * where every owner's run ends, how many entries there are, and the row of
 * slots they are laid in. Its three kernels, in their order:
 *   runs_ends    -- an inclusive prefix sum of the counts, so owner i's run
 *                   covers ends[i] - counts[i] up to, not including, ends[i];
 *   runs_entries -- how many entries the runs hold, at least one so that
 *                   the row is never empty: max(total, 1);
 *   runs_slots   -- the row of `entries` slots, every one -1.
 * Counts and ends are uint32 (ends wrap like the scan; a meaningful layout
 * keeps the total below 2^31). Returns entries; ends may be counts.
 * ---------------------------------------------------------------------- */

uint32_t oracle_runs_layout_u32(const uint32_t *counts, uint64_t n, uint32_t *ends)
{
    /* runs_ends */
    uint32_t run = 0;
    for (uint64_t i = 0; i < n; ++i) {
        run += counts[i];
        ends[i] = run;
    }
    /* runs_entries */
    return run > 0 ? run : 1u;
}

/*
 * The graph's description fills the slots (after runs_slots made them -1)
 * with a scatter over the owners that walks each owner's count, putting its
 * entry of rank r at ends[i] - counts[i] + r, with max. Here the value put
 * is the owner's index i, so slot e ends up holding the owner of entry e:
 * owner(e, ends). A slot no run reaches keeps its -1. `slots` holds
 * `entries` values; a write outside them is dropped.
 */
void oracle_runs_fill_owner(const uint32_t *counts, const uint32_t *ends, uint64_t n,
                            int32_t *slots, uint64_t entries)
{
    /* runs_slots */
    for (uint64_t e = 0; e < entries; ++e)
        slots[e] = -1;
    /* the scatter over the owners */
    for (uint64_t i = 0; i < n; ++i) {
        uint64_t start = (uint64_t)ends[i] - (uint64_t)counts[i];
        for (uint64_t r = 0; r < counts[i]; ++r) {
            uint64_t e = start + r;
            if (e >= entries)
                break; /* dropped, and so is the rest of this run */
            if ((int32_t)i > slots[e])
                slots[e] = (int32_t)i;
        }
    }
}

/* ------------------------------------------------------------------------
 * Compaction of values.  [CAIRN] "reduce and compact": `compact out for i
 * in n where p yield e` evaluates the test once per input, writes e for
 * each selected i, in order, to the front of out (capacity n), returns how
 * many it wrote, and leaves the rest of out unchanged. Here e = values[i]
 * and the test is flags[i] != 0, or, with no flags, values[i] != 0 (the
 * page's `where xs[i] > 0` on unsigned values).
 * ---------------------------------------------------------------------- */

uint64_t oracle_compact_values_u32(const uint32_t *values, const int32_t *flags, uint64_t n, uint32_t *out)
{
    uint64_t used = 0;
    for (uint64_t i = 0; i < n; ++i) {
        int keep = flags ? flags[i] != 0 : values[i] != 0;
        if (keep)
            out[used++] = values[i];
    }
    return used;
}

/* ------------------------------------------------------------------------
 * The same operators on uint64 rows.  [CAIRN] "reduce and compact": the
 * page's reductions run over u64 terms (u64(bytes[i]), mul_wrap(...)), and
 * add_wrap / mul_wrap wrap at 2^64 there. Exclusive and inclusive as in
 * oracle_scan_op_u32; returns the fold of all n.
 * ---------------------------------------------------------------------- */

static uint64_t oracle_apply64(int op, uint64_t x, uint64_t y)
{
    switch (op) {
    case 0: return x + y;
    case 1: return x * y;
    case 2: return x & y;
    case 3: return x | y;
    case 4: return x ^ y;
    case 5: return x < y ? x : y;
    default: return x > y ? x : y;
    }
}

static uint64_t oracle_identity64(int op)
{
    switch (op) {
    case 1: return 1u;
    case 2: case 5: return ~(uint64_t)0;
    default: return 0u;
    }
}

uint64_t oracle_scan_op_u64(int op, int inclusive, uint64_t *a, uint64_t n)
{
    uint64_t s = oracle_identity64(op);
    for (uint64_t j = 0; j < n; ++j) {
        uint64_t x = a[j];
        if (inclusive) {
            s = oracle_apply64(op, s, x);
            a[j] = s;
        } else {
            a[j] = s;
            s = oracle_apply64(op, s, x);
        }
    }
    return s;
}

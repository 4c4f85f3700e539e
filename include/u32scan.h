/*
 * u32scan.h -- C ABI of the GB300 (sm_103a) U32 scan library, libu32scan.so.
 *
 * Device-wide parallel prefix sums over arrays of 32-bit unsigned integers,
 * sums wrapping at 2^32, and the primitives built on them: segmented scan and
 * reduce over head-flagged segments, stream compaction (flags -> inclusive
 * offsets -> gathered indices -> count) and a stable LSD radix-sort
 * permutation of U32 keys.
 *
 * Conventions for every entry point below:
 *   - Pointers named as device pointers must point to memory the current
 *     CUDA device can access (cudaMalloc, torch tensors, managed memory),
 *     aligned to 4 bytes. 16-byte alignment is not required. Only the
 *     *_host scans take host pointers, and say so.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream). Results, totals and counts stay in device memory (the
 *     *_host scans write theirs to host memory).
 *   - The caller owns every buffer. The library allocates no memory and
 *     keeps no state between calls other than what lives in `ws` (and, for
 *     scan_exclusive_u32_noalloc, in that entry point's own static array).
 *   - `ws`/`ws_bytes` is caller-provided device workspace of at least
 *     u32scan_workspace_bytes(op, n) bytes (256-byte aligned). It must be
 *     zero-filled once before its first use (cudaMemset or
 *     u32scan_workspace_init); after that the library keeps it consistent
 *     itself, so it is reused across calls and shared between operations
 *     without clearing (the folds, the host-memory scans and small radix
 *     sorts, which keep other data in it, clear what they leave where other
 *     operations keep tile state before they return; a large radix sort
 *     keeps its buffers past that span). This holds for any
 *     number of calls: carry words are tagged with a per-workspace launch
 *     count whose tags repeat every 2^29 launches, and the launch that ends
 *     such a period zeroes the carry words (up to a few MiB of ws) before the
 *     next one starts. A workspace serves one call at a time: calls that
 *     share one workspace must be ordered (the same stream, or events).
 *   - Return value: U32SCAN_OK, or a negative status. Argument errors are
 *     found on the host before anything is launched; nothing is written
 *     then. U32SCAN_ECUDA reports a launch failure (cudaGetLastError).
 *     A device-side status (a carry wait that ran out of time) is reported
 *     by u32scan_check().
 *   - n == 0 is valid: nothing is read, and totals/counts are set to 0.
 */
#ifndef U32SCAN_H
#define U32SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (cudaStream_t), declared without
 * including any CUDA header. */
typedef struct CUstream_st *u32scan_stream_t;

#define U32SCAN_OK 0
#define U32SCAN_EINVAL (-1)     /* a null pointer with n > 0, misalignment, n too large */
#define U32SCAN_EWORKSPACE (-2) /* ws null or ws_bytes below u32scan_workspace_bytes */
#define U32SCAN_ECUDA (-3)      /* a CUDA runtime error (launch, memset, sync) */
#define U32SCAN_ETIMEOUT (-4)   /* device: a wait for a predecessor tile's carry timed out */

/* Operators for scan_u32_op: the integer operators of the CAIRN
 * "Concurrency" page's reduce and scan (add_wrap, mul_wrap, &, |, ^, min,
 * max), on uint32. Identities: 0, 1, all ones, 0, 0, all ones, 0. */
#define U32SCAN_ADD 0
#define U32SCAN_MUL 1
#define U32SCAN_AND 2
#define U32SCAN_OR 3
#define U32SCAN_XOR 4
#define U32SCAN_MIN 5
#define U32SCAN_MAX 6

/* Operation codes for u32scan_workspace_bytes. */
#define U32SCAN_OP_SCAN 1      /* scan_exclusive_u32, scan_inclusive_u32 */
#define U32SCAN_OP_SEGSCAN 2   /* segscan_inclusive_u32, segreduce_u32 (and _u8heads) */
#define U32SCAN_OP_COMPACT 3   /* compact_indices_u32, compact_values_u32 */
#define U32SCAN_OP_RADIX 4     /* radix_sort_perm_u32, radix_sort_u32 */
#define U32SCAN_OP_RUNS 5      /* runs_layout_u32 (runs_owner_u32 needs none) */
#define U32SCAN_OP_SCAN64 6    /* scan_u64_op */
#define U32SCAN_OP_SCAN_HOST 7 /* scan_exclusive_u32_host, scan_inclusive_u32_host */
#define U32SCAN_OP_REDUCE 8    /* reduce_u32_op (the same size for every n) */

/* Bytes of device workspace an operation needs for n elements (a multiple
 * of 256, at least 256). Returns 0 for an unknown op. Pure host function. */
size_t u32scan_workspace_bytes(int op, size_t n);

/* Zero-fill a workspace (cudaMemsetAsync on `stream`). */
int u32scan_workspace_init(void *ws, size_t ws_bytes, u32scan_stream_t stream);

/* Wait for `stream`, then read and clear the device-side status that the
 * calls using `ws` left: U32SCAN_OK, or U32SCAN_ETIMEOUT when a tile gave up
 * waiting for its predecessor's carry or a block gave up waiting for a tile's
 * bulk copy (the results of that call are then wrong). After a timeout,
 * zero-fill the workspace again (u32scan_workspace_init) before reusing it:
 * a launch whose blocks stopped early may leave its tile counter unreset.
 * U32SCAN_ECUDA if the synchronisation or the read fails. */
int u32scan_check(void *ws, u32scan_stream_t stream);

/* A static string for a status code. */
const char *u32scan_strerror(int status);

/* Library version, MAJOR * 10000 + MINOR * 100 + PATCH. */
int u32scan_version(void);

/*
 * Exclusive scan, in place.
 * Source: "scan.bend source" (bendlib), section API, `exclusive`: a[j]
 * becomes a[0] + .. + a[j-1] (a[0] becomes 0) and the call returns the
 * total a[0] + .. + a[n-1]; header comment: sums wrap at 2^32. Also the
 * CAIRN "Concurrency" page, section "scan" (`scan + exclusive`, binds the
 * total).
 *   data  device, uint32_t[n], read and overwritten with the scan.
 *   n     element count; any n up to 2^32 - 1.
 *   total device, one uint32_t written with the wrapped total; may be NULL.
 * Errors: EINVAL if data is NULL with n > 0, if data or total is not 4-byte
 * aligned, or n >= 2^32; EWORKSPACE; ECUDA.
 */
int scan_exclusive_u32(uint32_t *data, size_t n, uint32_t *total,
                       void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Inclusive scan, in place: a[j] becomes a[0] + .. + a[j], wrapping.
 * Source: "scan.bend source", section API, `inclusive`; CAIRN "scan"
 * (`scan + out`, out[i] = e(0) + .. + e(i)). Arguments and errors as
 * scan_exclusive_u32.
 */
int scan_inclusive_u32(uint32_t *data, size_t n, uint32_t *total,
                       void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * The two scans of one piece of a longer array: the piece starts after a
 * carry-in, the wrapped sum of everything before it (a device word, so that
 * it can come from an earlier kernel or a collective without a host round
 * trip). Source: "scan.bend source", section Driver (each block is rescanned
 * from its base, the scan of the block sums before it) and section API; one
 * level up, the pieces are the shards of an array split across GPUs.
 *   data, n, ws, ws_bytes, stream  as scan_exclusive_u32.
 *   carry_in  device, one uint32_t (4-byte aligned), or NULL for 0:
 *             exclusive: data[j] = carry_in + data[0] + .. + data[j-1];
 *             inclusive: through data[j].
 *   total     device, one uint32_t or NULL: carry_in + data[0] + .. +
 *             data[n-1] (wrapping); must not be carry_in itself (the block
 *             holding the first tile may read the carry-in after the last
 *             tile has written the total).
 * Errors: EINVAL (as scan_exclusive_u32, a misaligned carry_in, total ==
 * carry_in), EWORKSPACE, ECUDA.
 */
int scan_exclusive_u32_carry(uint32_t *data, size_t n, const uint32_t *carry_in, uint32_t *total,
                             void *ws, size_t ws_bytes, u32scan_stream_t stream);
int scan_inclusive_u32_carry(uint32_t *data, size_t n, const uint32_t *carry_in, uint32_t *total,
                             void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * The fold of an array under one of U32SCAN_ADD .. U32SCAN_MAX, reading it
 * once (4 bytes an element) and writing nothing else. Source: the CAIRN
 * "Concurrency" page, section "reduce and compact" (`reduce` with add_wrap,
 * mul_wrap, &, |, ^, min, max; sums and products wrap at 2^32). Every such
 * operator is associative and commutative, so the result does not depend on
 * the order in which the device folds.
 *   op        U32SCAN_ADD .. U32SCAN_MAX.
 *   data      device, uint32_t[n], 4-byte aligned, read only.
 *   n         element count, below 2^62.
 *   total     device, one uint32_t (4-byte aligned): the fold (the
 *             operator's identity when n == 0).
 *   ws, ws_bytes  u32scan_workspace_bytes(U32SCAN_OP_REDUCE, n) bytes (a
 *             few KiB, the same for every n), 256-byte aligned, zero-filled
 *             once; shared with the other operations like any workspace.
 * Errors: EINVAL (unknown op, null data with n > 0, null total, misaligned
 * pointers), EWORKSPACE, ECUDA.
 */
int reduce_u32_op(int op, const uint32_t *data, size_t n, uint32_t *total,
                  void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * The number of non-zero elements, read once: the count of a compaction
 * without its offsets. Source: the "parallel" package reference (entelechy
 * docs), graph `compact`: compact_total is the number of kept elements, and a
 * non-zero flag keeps its element.
 *   data   device, uint32_t[n] (int32 flags may be passed as is), read only.
 *   n      element count, below 2^62; count wraps at 2^32.
 *   count  device, one uint32_t: the number of data[i] != 0 (0 when n == 0).
 *   ws, ws_bytes  as reduce_u32_op (U32SCAN_OP_REDUCE).
 * Errors: as reduce_u32_op.
 */
int count_nonzero_u32(const uint32_t *data, size_t n, uint32_t *count,
                      void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * The same two scans of an array in HOST memory, with the result written to
 * host memory. Source: as scan_exclusive_u32 / scan_inclusive_u32
 * ("scan.bend source", section API; CAIRN "scan"); the pages' arrays live in
 * device memory, and these entry points carry a host array through the
 * device scan. The array moves in chunks through staging slots in `ws`:
 * copies in, chunk scans and copies out overlap on three streams (two
 * created inside the call, released when their work completes), and each
 * chunk's scan starts from the wrapped sum of the chunks before it.
 *   host_in     HOST, uint32_t[n], page-locked (cudaHostAlloc, cudaMallocHost,
 *               cudaHostRegister; torch pin_memory), read only.
 *   host_out    HOST, uint32_t[n], page-locked: the scan. May be host_in
 *               itself (in place); must not overlap it otherwise.
 *   n           element count, any n below 2^62.
 *   host_total  HOST, one page-locked uint32_t, or NULL: the wrapped total.
 *   ws, ws_bytes  device, u32scan_workspace_bytes(U32SCAN_OP_SCAN_HOST, n)
 *               bytes (at most 128 MiB of staging plus the scan's carry
 *               words), 256-byte aligned, zero-filled once.
 *   stream      the scans run on it; the call returns at once, and the
 *               outputs are complete when `stream` reaches the point of the
 *               call (cudaStreamSynchronize(stream) waits for them).
 * Errors: EINVAL (null in/out with n > 0, pointers not 4-byte aligned, host
 * buffers not page-locked, partial overlap of in and out, total overlapping
 * either, n >= 2^62), EWORKSPACE, ECUDA (a stream, event, copy or launch
 * failed; work already queued still completes before later work on
 * `stream`). A carry-wait timeout is reported by u32scan_check(ws, stream).
 */
int scan_exclusive_u32_host(const uint32_t *host_in, uint32_t *host_out, size_t n, uint32_t *host_total,
                            void *ws, size_t ws_bytes, u32scan_stream_t stream);
int scan_inclusive_u32_host(const uint32_t *host_in, uint32_t *host_out, size_t n, uint32_t *host_total,
                            void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Scan in place under any of the U32SCAN_ADD .. U32SCAN_MAX operators.
 * Source: CAIRN "Concurrency" page, section "scan" ("the operators are
 * those of reduce": add_wrap, mul_wrap, &, |, ^, min, max; `scan max` is
 * printed there) and section "reduce and compact".
 *   op         U32SCAN_ADD .. U32SCAN_MAX.
 *   inclusive  0: data[j] = e . data[0] . .. . data[j-1] (e the identity);
 *              1: through data[j].
 *   total      device, one uint32_t or NULL: the fold of all n elements
 *              (the identity when n == 0).
 *   data, n, ws, ws_bytes, stream: as scan_exclusive_u32 (workspace
 *              u32scan_workspace_bytes(U32SCAN_OP_SCAN, n)).
 * U32SCAN_ADD gives exactly scan_exclusive_u32 / scan_inclusive_u32.
 * Errors: EINVAL for an unknown op, and as scan_exclusive_u32.
 */
int scan_u32_op(int op, int inclusive, uint32_t *data, size_t n, uint32_t *total,
                void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * The same scans on uint64 rows. Source: CAIRN "Concurrency" page, sections
 * "reduce and compact" (integer operators; its examples reduce u64 terms)
 * and "scan". add_wrap and mul_wrap wrap at 2^64.
 *   op, inclusive  as scan_u32_op.
 *   data     device, uint64_t[n], 8-byte aligned; scanned in place.
 *   n        element count, below 2^32.
 *   total    device, one uint64_t (8-byte aligned) or NULL: the fold of all n
 *            elements (the identity when n == 0).
 *   ws, ws_bytes  u32scan_workspace_bytes(U32SCAN_OP_SCAN64, n) bytes,
 *            256-byte aligned, zero-filled once; reusable in stream order.
 * Errors: EINVAL (unknown op, null data with n > 0, misaligned pointers,
 * n >= 2^32), EWORKSPACE, ECUDA; a look-back timeout as the u32 scans'.
 */
int scan_u64_op(int op, int inclusive, uint64_t *data, size_t n, uint64_t *total,
                void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Segmented inclusive scan, in place, optionally with per-segment sums.
 * Source: "Futhark.Pass.ExtractKernels.Segmented" (regularSegmentedScan;
 * regularSegmentedRedomap for the per-segment reduce, "a single value per
 * segment"). A non-zero head_flags[j] opens a segment at j; index 0 always
 * opens one. data[j] becomes data[h] + .. + data[j] (mod 2^32), h the last
 * head at or before j.
 *   data         device, uint32_t[n], read and overwritten.
 *   head_flags   device, int32_t[n], read only.
 *   n            element count, below 2^32.
 *   seg_sums     device, uint32_t[seg_capacity] or NULL: seg_sums[k] gets
 *                the wrapped sum of segment k (segments in index order);
 *                segments k >= seg_capacity are not written.
 *   seg_capacity slots in seg_sums (ignored when seg_sums is NULL).
 *   nseg         device, one uint32_t or NULL: the number of segments
 *                (0 when n == 0), even when it exceeds seg_capacity.
 *   ws, ws_bytes u32scan_workspace_bytes(U32SCAN_OP_SEGSCAN, n) bytes.
 * data and head_flags need 4-byte alignment; when their addresses differ
 * mod 16 the kernel falls back to scalar loads (correct, slower).
 * Errors: EINVAL (null data/flags with n > 0, misaligned pointers,
 * n >= 2^32), EWORKSPACE, ECUDA.
 */
int segscan_inclusive_u32(uint32_t *data, const int32_t *head_flags, size_t n,
                          uint32_t *seg_sums, size_t seg_capacity, uint32_t *nseg,
                          void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Per-segment reduce: the sums and count of segscan_inclusive_u32 without
 * writing the scan (data is only read). Source as above
 * (regularSegmentedRedomap). At least one of seg_sums and nseg must be
 * non-NULL (EINVAL otherwise); other arguments and errors as
 * segscan_inclusive_u32.
 */
int segreduce_u32(const uint32_t *data, const int32_t *head_flags, size_t n,
                  uint32_t *seg_sums, size_t seg_capacity, uint32_t *nseg,
                  void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * The segmented scan of one array split into pieces (one per rank, say):
 * each piece is scanned on its own with segscan_inclusive_u32, then summed
 * up, the summaries combined in piece order, and each piece fixed from its
 * carry-in. Source: "Futhark.Pass.ExtractKernels.Segmented"
 * (regularSegmentedScan) for the operation; the scan.bend source's Driver
 * (block sums, their scan, each block finished from its base) for the
 * composition. The segmented operator over a piece is (has a head, the
 * segmented value at its end); the value flowing into piece r + 1 is piece
 * r's tail when piece r holds a head, else the value flowing into piece r
 * plus that tail. Only the elements before a piece's first head depend on
 * it.
 *
 * segscan_piece_summary_u32: one piece's summary, three uint32_t at
 * `summary` (device): whether the piece holds a head (any non-zero flag,
 * element 0 included), the scanned value of its last element, and its
 * segment count as a piece of the whole array (segments that start in it).
 *   scanned      device, uint32_t[n]: the piece after segscan_inclusive_u32.
 *   head_flags   device, int32_t[n]: the piece's flags.
 *   nseg         device, one uint32_t: the count segscan_inclusive_u32 gave.
 *   first_opens  non-zero for the first piece (its element 0 opens the
 *                array's first segment), 0 for the others.
 *   n == 0 gives (0, 0, 0).
 * segscan_piece_carries_u32: from the g pieces' summaries in piece order
 * (device, uint32_t[3 g]), each piece's carry-in (device, uint32_t[g]; the
 * first is 0) and the whole array's segment count (device, one uint32_t, or
 * NULL).
 * segscan_fix_u32: adds the carry-in (device, one uint32_t) to the elements
 * of the scanned piece `data` before its first head (all of them when it
 * has none); `ws`: any workspace of the library (at least its 256-byte
 * header), zero-filled once; the call keeps it so.
 * All three are asynchronous on `stream`. Errors: EINVAL (null pointers the
 * call needs, misaligned pointers, n >= 2^32), EWORKSPACE, ECUDA.
 */
int segscan_piece_summary_u32(const uint32_t *scanned, const int32_t *head_flags, size_t n,
                              const uint32_t *nseg, int first_opens, uint32_t *summary,
                              u32scan_stream_t stream);
int segscan_piece_carries_u32(const uint32_t *summaries, size_t g, uint32_t *carries, uint32_t *nseg_total,
                              u32scan_stream_t stream);
int segscan_fix_u32(uint32_t *data, const int32_t *head_flags, size_t n, const uint32_t *carry,
                    void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * The same two operations with one byte per head flag: a non-zero byte at j
 * opens a segment at j (the entelechy reading of a flag: non-zero is set).
 * Arguments, results, workspace (U32SCAN_OP_SEGSCAN) and errors as in
 * segscan_inclusive_u32 and segreduce_u32, except that head_flags is a
 * device uint8_t[n] with no alignment requirement. The flags stream by bulk
 * copy when (head_flags - (data mod 16) / 4) is 16-byte aligned (so for
 * two buffers of the same 16-byte phase in elements, e.g. fresh
 * allocations); otherwise by plain loads, with the same results.
 */
int segscan_inclusive_u32_u8heads(uint32_t *data, const uint8_t *head_flags, size_t n,
                                  uint32_t *seg_sums, size_t seg_capacity, uint32_t *nseg,
                                  void *ws, size_t ws_bytes, u32scan_stream_t stream);
int segreduce_u32_u8heads(const uint32_t *data, const uint8_t *head_flags, size_t n,
                          uint32_t *seg_sums, size_t seg_capacity, uint32_t *nseg,
                          void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Stream compaction: flags -> inclusive offsets -> gathered indices -> count.
 * Source: the "parallel" package reference (entelechy docs), graph
 * `compact`: compact_offsets (inclusive prefix sum, a kept element at i
 * belongs at offsets[i] - 1), compact_gather (each kept index written where
 * its rank says), compact_blank (an unfilled slot holds -1), compact_total
 * (the count as a row of one). A non-zero flag keeps its element.
 *   flags    device, int32_t[n], read only.
 *   n        element count, below 2^31.
 *   offsets  device, int32_t[n] or NULL: offsets[i] = number of non-zero
 *            flags in flags[0..i].
 *   indices  device, int32_t[n]: the kept indices in increasing order at the
 *            front, -1 in every slot after them. Every slot is written.
 *   count    device, one int32_t or NULL: the number of kept elements.
 *   ws, ws_bytes  u32scan_workspace_bytes(U32SCAN_OP_COMPACT, n) bytes.
 * All pointers need 4-byte alignment; offsets is written with 16-byte
 * stores when it has flags' alignment mod 16, else with 4-byte stores.
 * Errors: EINVAL (null flags or indices with n > 0, misaligned pointers,
 * n >= 2^31), EWORKSPACE, ECUDA.
 */
int compact_indices_u32(const int32_t *flags, size_t n, int32_t *offsets,
                        int32_t *indices, int32_t *count,
                        void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Compaction of values. Source: the CAIRN "Concurrency" page, "reduce and
 * compact": `compact out for i in n where p yield e` writes e for each
 * selected i, in order, to the front of out (capacity n), returns how many
 * it wrote and leaves the rest of out unchanged. Here e = values[i].
 *   values   device, uint32_t[n], read only.
 *   flags    device, int32_t[n] or NULL: element i is kept when flags[i] != 0;
 *            with NULL, when values[i] != 0 (the page's `where xs[i] > 0`).
 *   out      device, uint32_t[n]: the kept values in order at the front;
 *            out[count..n) is not written. Must not overlap values or flags.
 *   count    device, one int32_t or NULL: the number of kept elements.
 *   ws, ws_bytes  u32scan_workspace_bytes(U32SCAN_OP_COMPACT, n) bytes.
 * All pointers need 4-byte alignment. Flags stream by bulk copy when they
 * have values' alignment mod 16, else by plain loads (same results).
 * Errors: EINVAL (null values or out with n > 0, misaligned pointers,
 * n >= 2^31, out overlapping values or flags), EWORKSPACE, ECUDA.
 */
int compact_values_u32(const uint32_t *values, const int32_t *flags, size_t n, uint32_t *out,
                       int32_t *count, void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * compact_indices_u32 of one piece of a longer flag array: what lies before
 * the piece comes in as two device words (so that they can come from a
 * collective without a host round trip), and the piece's results are its
 * part of the whole array's. Source: as compact_indices_u32; the pieces
 * compose as the scan.bend source's blocks do (section Driver): a piece's
 * offsets start from the kept count before it.
 *   kept_before  device, one int32_t or NULL for 0: kept elements before the
 *                piece; offsets[i] = kept_before + kept in flags[0..i].
 *   first_index  device, one int32_t or NULL for 0: the whole array's index
 *                of flags[0]; the kept indices written are whole-array
 *                indices (first_index + i).
 *   flags, n, offsets, indices, count, ws, ws_bytes, stream: as
 *                compact_indices_u32; indices and count are the piece's own
 *                (its kept indices in order at the front, -1 after them, and
 *                its kept count). The whole array's compacted indices are the
 *                pieces' fronts one after another. Whole-array indices must
 *                stay below 2^31.
 * Errors: as compact_indices_u32, and EINVAL for a misaligned kept_before or
 * first_index.
 */
int compact_indices_u32_carry(const int32_t *flags, size_t n, const int32_t *kept_before,
                              const int32_t *first_index, int32_t *offsets, int32_t *indices, int32_t *count,
                              void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Stable LSD radix-sort permutation of U32 keys.
 * Source: the "parallel" package reference (entelechy docs), graph `sort`
 * (the permutation that orders the keys, least significant bit first;
 * sort_zeros / sort_place: a stable pass per bit), and the CAIRN
 * "Concurrency" page, section "scan" (std.sort.radix_sort places each
 * digit with an exclusive scan, so it is stable).
 *   keys   device, uint32_t[n], read only; all 32 bits, unsigned order.
 *   n      element count, below 2^31.
 *   perm   device, int32_t[n]: keys[perm[0]] <= keys[perm[1]] <= ..., equal
 *          keys in increasing index order (the unique stable permutation).
 *   ws, ws_bytes  u32scan_workspace_bytes(U32SCAN_OP_RADIX, n) bytes (about
 *          12 * n bytes: two key buffers and one index buffer; from n of
 *          about 700,000 on, plus about 8.4 MB before them, the span other
 *          operations' carry words can take, which the sort then need not
 *          clear).
 * Digits that are equal for every key are skipped; which passes run is
 * decided on the device, so the call is asynchronous like the others.
 * Errors: EINVAL (null keys or perm with n > 0, misaligned pointers,
 * n >= 2^31), EWORKSPACE, ECUDA.
 */
int radix_sort_perm_u32(const uint32_t *keys, size_t n, int32_t *perm,
                        void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Stable LSD radix sort of U32 keys, with the sorted keys as output: the
 * permutation passes of radix_sort_perm_u32, whose last pass also writes
 * the keys. Same source passages.
 *   keys      device, uint32_t[n], read only.
 *   keys_out  device, uint32_t[n]: the keys in non-decreasing order; must not
 *             overlap keys.
 *   perm      device, int32_t[n] or NULL: the stable permutation as in
 *             radix_sort_perm_u32 (keys_out[i] = keys[perm[i]]). NULL sorts
 *             the keys alone and moves no indices.
 *   ws, ws_bytes  u32scan_workspace_bytes(U32SCAN_OP_RADIX, n) bytes.
 * Errors: EINVAL (null keys or keys_out with n > 0, misaligned pointers,
 * overlapping keys and keys_out, n >= 2^31), EWORKSPACE, ECUDA.
 */
int radix_sort_u32(const uint32_t *keys, size_t n, uint32_t *keys_out, int32_t *perm,
                   void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * Runs layout. Source: the "parallel" package reference (entelechy docs),
 * graph `runs` and its kernels runs_ends (the inclusive prefix sum of the
 * counts: owner i's run covers ends[i] - counts[i] up to ends[i]),
 * runs_entries (how many entries, at least one) and runs_slots (the row of
 * `entries` slots, every one -1).
 *   counts    device, uint32_t[n]: entries per owner; replaced in place by
 *             ends (sums wrap at 2^32; a meaningful layout keeps the total
 *             below 2^31).
 *   entries   device, uint32_t[1]: max(total, 1).
 *   slots     device, int32_t[slot_capacity] or NULL: slots[e] = -1 for e in
 *             [0, min(entries, slot_capacity)); the rest untouched.
 *   ws, ws_bytes  u32scan_workspace_bytes(U32SCAN_OP_RUNS, n) bytes.
 * Errors: EINVAL (null counts with n > 0, null entries, misaligned pointers,
 * n >= 2^31, slot_capacity >= 2^32, entries or slots overlapping counts or
 * each other), EWORKSPACE, ECUDA; a look-back timeout as the scan's.
 */
int runs_layout_u32(uint32_t *counts, size_t n, uint32_t *entries, int32_t *slots, size_t slot_capacity,
                    void *ws, size_t ws_bytes, u32scan_stream_t stream);

/*
 * owner(e, ends) for every entry of a runs layout. Source: as runs_layout_u32,
 * function `owner(e: Int, ends: Rows<Int>) -> Int`; the page gives no text for
 * it, and the owner of entry e is read as the owner whose run holds e: the
 * least i with e < ends[i].
 *   ends      device, uint32_t[n], non-decreasing (runs_layout_u32's output).
 *   owner     device, int32_t[capacity]: owner[e] for e in [0, min(entries,
 *             capacity)), entries = max(ends[n-1], 1); the one slot of a
 *             layout with no entries (n = 0 or total 0) is -1. The rest is
 *             untouched. The row equals the layout's slots after the graph's
 *             fill scatter with each owner's index as the value.
 * No workspace. Errors: EINVAL (null ends with n > 0, null owner with
 * capacity > 0, misaligned pointers, n >= 2^31, capacity >= 2^32, owner
 * overlapping ends), ECUDA. Ends that are not non-decreasing give an
 * unspecified row, but every access stays inside ends[0, n) and
 * owner[0, capacity).
 */
int runs_owner_u32(const uint32_t *ends, size_t n, int32_t *owner, size_t capacity, u32scan_stream_t stream);

/*
 * Exclusive scan that allocates nothing and needs no workspace argument.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory (for instance code inside an allocator's
 * own callbacks, or a runtime that only lends out buffers it owns), so
 * they cannot provide the workspace scan_exclusive_u32 needs.
 *   data, n, total, stream: as scan_exclusive_u32; n at most 2^31.
 * Scratch: a fixed device array inside this library (about 4 MiB, held on
 * every GPU that loads the library until the process exits). The first
 * call on each device looks up that array's device address
 * (cudaGetSymbolAddress) with the device current; make that first call
 * before any stream capture. Each call enqueues the scan kernel alone on
 * `stream`; it calls no cudaMalloc, cudaFree or memset. The array keeps
 * its state between calls: each launch leaves it ready for the next.
 * All calls share the one array: calls that overlap on the GPU (different
 * streams, or different host threads without ordering) race and give wrong
 * results. Order them, e.g. on one stream.
 * Errors: EINVAL for n > 2^31 (the scratch limit) and as scan_exclusive_u32;
 * ECUDA if the set-up or a launch fails. A carry-wait timeout is recorded
 * in the array's status word: read it with u32scan_check_noalloc.
 */
int scan_exclusive_u32_noalloc(uint32_t *data, size_t n, uint32_t *total,
                               u32scan_stream_t stream);

/*
 * The device-side status of the allocation-free scan (no counterpart on the
 * pages): waits for `stream`, then reads and clears the status word of the
 * library's fixed array, as u32scan_check does for a workspace. Returns
 * U32SCAN_OK, or U32SCAN_ETIMEOUT when a call since the last check gave up
 * waiting (its results are then wrong; the array is then zero-filled on
 * `stream` and waited for, so later calls start afresh); U32SCAN_ECUDA if
 * the set-up, the synchronisation, the read or the fill fails. Allocates
 * nothing.
 */
int u32scan_check_noalloc(u32scan_stream_t stream);

/*
 * Test hook for the bounded carry wait (no counterpart on the pages; the
 * Relay page names the hazard it guards against: a tile waiting on a
 * predecessor that never hands its carry on). Runs scan_exclusive_u32,
 * except that tile `skip_tile` of the launch never publishes its carry,
 * so the tiles after it wait `limit_ns` nanoseconds, give up, and the next
 * u32scan_check() on `ws` returns U32SCAN_ETIMEOUT. The results are then
 * wrong by design; nothing else is affected, and `ws` stays usable.
 */
int u32scan_test_scan_skip_publish(uint32_t *data, size_t n, uint32_t *total,
                                   void *ws, size_t ws_bytes,
                                   unsigned int skip_tile,
                                   unsigned long long limit_ns,
                                   u32scan_stream_t stream);

/*
 * The same test hook for the segmented scan's two carry words (segmented
 * value and head count): runs segscan_inclusive_u32 (with or without
 * `seg_sums`), except that tile `skip_tile` of the launch publishes neither
 * word, so the tiles after it that need them wait `limit_ns` nanoseconds,
 * give up, and the next u32scan_check() on `ws` returns U32SCAN_ETIMEOUT.
 * The results are then wrong by design; `ws` stays usable. Tiles hold
 * 10240 elements with these int32 flags.
 */
int u32scan_test_segscan_skip_publish(uint32_t *data, const int32_t *head_flags, size_t n,
                                      uint32_t *seg_sums, size_t seg_capacity, uint32_t *nseg,
                                      void *ws, size_t ws_bytes,
                                      unsigned int skip_tile,
                                      unsigned long long limit_ns,
                                      u32scan_stream_t stream);

/*
 * The same test hook for the allocation-free scan (no counterpart on the
 * pages): runs scan_exclusive_u32_noalloc with tile `skip_tile` never
 * publishing its carry, so the next u32scan_check_noalloc() returns
 * U32SCAN_ETIMEOUT. Tiles hold 2048 elements below 2^19 elements, 16384
 * from there. The results are then wrong by design; later calls are not
 * affected.
 */
int u32scan_test_noalloc_skip_publish(uint32_t *data, size_t n, uint32_t *total, unsigned int skip_tile,
                                      unsigned long long limit_ns, u32scan_stream_t stream);

/*
 * Test hook (no counterpart on the pages): sets the launch count of the
 * allocation-free scan's fixed array, ordered on `stream`, so that a test
 * can reach the end of a tag period (2^29 launches) without making them.
 */
int u32scan_test_noalloc_set_epoch(unsigned int epoch, u32scan_stream_t stream);

/*
 * Seeded synthetic input, drawn on the device (no counterpart on the pages,
 * which measure on synthetic inputs only): out[i] = u32(seed, stream,
 * start + i) for i < n, where u32 is counter-based SplitMix64 (S. Vigna's
 * public-domain mixer): the high 32 bits of mix((seed << 40) | (stream << 32)
 * | index), the same numbers as the host generator in
 * u32_prefix_scan_gb300/inputs.py. Lets a caller draw a large input in
 * device memory instead of copying it from the host.
 *   out:    device, n words, 4-byte aligned; written, caller-owned.
 *   seed:   below 2^24; stream: below 256; start + n at most 2^32.
 * Asynchronous on `stream`. Errors: EINVAL for a null or misaligned `out`
 * with n > 0 or an argument out of range; ECUDA if the launch fails. n = 0
 * does nothing.
 */
int u32scan_fill_splitmix_u32(uint32_t *out, size_t n, uint32_t seed, uint32_t stream, size_t start,
                              u32scan_stream_t cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* U32SCAN_H */

// segscan.cu -- segmented inclusive U32 scan and per-segment reduce.
//
// Source: "Futhark.Pass.ExtractKernels.Segmented": regularSegmentedScan
// names the segmented scan; regularSegmentedRedomap reduces every segment
// "until there is only a single value per segment". Segments are marked by
// head flags: a non-zero flag at j opens a segment at j, and index 0 always
// opens one. Flags are int32 (segscan_inclusive_u32, segreduce_u32) or one
// byte each (the _u8heads entry points: 9 bytes per element for the scan
// instead of 12). The scan gives out[j] = a[h] + .. + a[j] (mod 2^32), h
// the last head at or before j; the reduce gives one wrapped sum per
// segment, in segment order, and the segment count.
//
// The page's two strategies (one group per segment for long segments,
// several segments per group for short ones, chosen at run time) are prior
// art: here one single-pass kernel serves every segment-length mix, because
// the segmented operator (head, sum) is associative and carries across
// tiles like a plain sum. A tile's carry stops at the nearest earlier tile
// that holds a head.
//
// Kernel: persistent, one block per SM, the same one-tile software pipeline
// as the plain scan (scan.cu): two 1-D bulk copies per tile (values and head
// flags) into a ring of shared-memory stages; each round reads and scans
// the next tile and publishes its aggregate, then walks the current tile's
// look-back, adds the carry and stores. Per tile the look-back carries two
// words (internal.cuh): the segmented value and the running head count; the
// head count gives every segment end its index into the sums.
//
// Layout inside a tile: warp w owns the w-th run of 128 * V elements; in
// round r (of V / Q) lane l holds the E = 4 Q consecutive elements at
// 32 E r + E l of that run, as Q u32x4. Head flags become one bit per
// element (bit 4 i + c for component c of the lane's i-th u32x4); byte flags
// are read four to a word and tested bytewise. Each round costs one warp-wide
// segmented scan, so more elements a lane a round means fewer per element.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

#ifndef U32SCAN_S_LOOKA
#define U32SCAN_S_LOOKA 1  // look-back words a lane per round trip: segmented value
#endif
#ifndef U32SCAN_S_LOOKB
#define U32SCAN_S_LOOKB 1  // and head count
#endif

namespace u32scan {

constexpr unsigned int kNoHead = 0xffffffffu;

// Component c of a u32x4.
__device__ __forceinline__ unsigned int comp(const uint4 &v, int c) {
    return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}
__device__ __forceinline__ void set_comp(uint4 &v, int c, unsigned int a) {
    if (c == 0) v.x = a; else if (c == 1) v.y = a; else if (c == 2) v.z = a; else v.w = a;
}

template <int THREADS, int V, int Q, int S, bool WRITE_SCAN, bool WANT_SUMS, typename F>
__global__ void __launch_bounds__(THREADS, 512 / THREADS)
segscan_u32_persistent(uint32_t *__restrict__ data, const F *__restrict__ flags, unsigned long long n,
                       uint32_t *seg_sums, unsigned long long seg_cap, uint32_t *nseg, WsHeader *hdr,
                       unsigned long long *desc2, unsigned int n_tiles, unsigned int head, int streams_aligned,
                       unsigned int skip_tile, unsigned long long limit_ns) {
    constexpr int WARPS = THREADS / 32;
    constexpr unsigned int CHUNK = 128 * V;  // elements per warp
    constexpr unsigned int TILE = THREADS * V * 4;
    // A lane takes E = 4 Q consecutive elements a round (Q u32x4), R rounds.
    constexpr int R = V / Q, E = 4 * Q;
    constexpr unsigned int kEMask = (1u << E) - 1u;
    static_assert(V % Q == 0 && E <= 16, "whole rounds of u32x4");
    // x[i] holds lane-local elements 4i .. 4i + 3: round i / Q, part i % Q;
    // u4_off(i) is its offset from the lane's first element, in u32x4.
    auto u4_off = [](int i) -> unsigned int { return 32u * Q * (unsigned int)(i / Q) + (unsigned int)(i % Q); };
    constexpr unsigned int TILE_BYTES = TILE * 4;  // values
    constexpr unsigned int FLAG_BYTES = TILE * (unsigned int)sizeof(F);
    constexpr unsigned int STAGE_U4 = (TILE_BYTES + FLAG_BYTES) / 16;
    static_assert(WARPS <= 32 && 4 * V <= 32, "one lane per warp; head bits fit in a word");
    static_assert(sizeof(F) == 4 || sizeof(F) == 1, "int32 or byte head flags");
    extern __shared__ __align__(128) uint4 stage_buf[];  // S stages of [values | flags]
    __shared__ __align__(8) unsigned long long bar[S];
    __shared__ unsigned int s_tile[S];
    __shared__ unsigned int s_wval[2][WARPS], s_wcnt[2][WARPS], s_whas[2][WARPS];
    // Head bit of each warp's first element, read after barrier B by the
    // previous warp; three slots, so a warp already reading the next tile
    // never overwrites the slot of a tile still being stored.
    __shared__ unsigned int s_wfirst[3][WARPS];
    __shared__ unsigned int s_bval[WARPS], s_bcnt[WARPS], s_nexthead;
    __shared__ unsigned int s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned int last_draw = n_tiles + (unsigned int)S * gridDim.x - 1u;
    uint32_t *vdata = reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(data) - 4ull * head);
    const F *vflags = reinterpret_cast<const F *>(reinterpret_cast<uintptr_t>(flags) - sizeof(F) * head);
    const bool producer = threadIdx.x == THREADS - 32;
    unsigned int latest_parity = 0;

    auto tile_full = [&](unsigned int id) {
        const unsigned long long v0 = (unsigned long long)id * TILE;
        return streams_aligned && v0 >= head && v0 + TILE <= head + n;
    };
    auto tile_range = [&](unsigned int id, unsigned int &lo, unsigned int &hi) {
        const unsigned long long v0 = (unsigned long long)id * TILE;
        lo = v0 < head ? (unsigned int)(head - v0) : 0u;
        const unsigned long long left = head + n - v0;
        hi = left < TILE ? (unsigned int)left : TILE;
    };
    auto issue = [&](int st) {  // producer only
        const unsigned int id = atom_add_acq_rel(&hdr->counter, 1u);
        if (id == last_draw) {
            st_relaxed_u32(&hdr->counter, 0u);
            st_relaxed_u32(&hdr->epoch, s_epoch + 1u);
        }
        s_tile[st] = id;
        const unsigned int b = smem_u32(&bar[st]);
        if (id < n_tiles && tile_full(id)) {
            const unsigned long long v0 = (unsigned long long)id * TILE;
            mbar_arrive_expect_tx(b, TILE_BYTES + FLAG_BYTES);
            bulk_load(smem_u32(stage_buf + st * STAGE_U4), vdata + v0, TILE_BYTES, b);
            bulk_load(smem_u32(stage_buf + st * STAGE_U4 + TILE / 4), vflags + v0, FLAG_BYTES, b);
        } else {
            mbar_arrive(b);  // nothing to copy: a partial tile reads global memory, a past-the-end draw stops
        }
    };

    if (producer) {
#pragma unroll
        for (int st = 0; st < S; ++st) mbar_init(smem_u32(&bar[st]), 1u);
        fence_mbar_init();
        fence_proxy_async_smem();
        s_epoch = ld_relaxed_u32(&hdr->epoch);
#pragma unroll
        for (int st = 0; st < S; ++st) issue(st);
    }
    __syncthreads();
    const unsigned long long tag = tag_of(s_epoch);
    const unsigned int li0 = (unsigned int)warp * CHUNK + (unsigned int)E * (unsigned int)lane;
    volatile unsigned int *vs_tile = s_tile;

    // Read draw u into registers (values x, head bits hb), scan it within
    // each warp and leave the warp aggregates in slot u & 1. Returns the
    // tile, or n_tiles and above past the end / on a timeout.
    auto read_tile = [&](unsigned int u, uint4 (&x)[V], unsigned int &hb, unsigned int &pfirst,
                         unsigned int (&cl)[R]) -> unsigned int {
        const int st = (int)(u % S);
        if (!mbar_wait_bounded(smem_u32(&bar[st]), (u / S) & 1u, limit_ns)) {
            report_timeout(hdr, 0xfffffffeu);
            return n_tiles + 1u;
        }
        const unsigned int t = vs_tile[st];
        if (t >= n_tiles) return n_tiles;
        const unsigned long long tile_v0 = (unsigned long long)t * TILE;
        hb = 0;
        if (tile_full(t)) {
            const uint4 *sv = stage_buf + st * STAGE_U4 + (li0 >> 2);
            if constexpr (sizeof(F) == 4) {
                const int4 *sf = reinterpret_cast<const int4 *>(stage_buf + st * STAGE_U4 + TILE / 4) + (li0 >> 2);
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    x[i] = sv[u4_off(i)];
                    const int4 f = sf[u4_off(i)];
                    hb |= ((f.x != 0) | ((f.y != 0) << 1) | ((f.z != 0) << 2) | ((f.w != 0) << 3)) << (4 * i);
                }
            } else {
                // four byte flags in one word: byte c non-zero -> bit c of a nibble
                const unsigned int *sf = reinterpret_cast<const unsigned int *>(stage_buf + st * STAGE_U4 + TILE / 4) +
                                         (li0 >> 2);
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    x[i] = sv[u4_off(i)];
                    const unsigned int m = __vcmpne4(sf[u4_off(i)], 0u) & 0x08040201u;
                    hb |= ((m * 0x01010101u) >> 24) << (4 * i);
                }
            }
        } else {
            unsigned int lo, hi;
            tile_range(t, lo, hi);
            const uint32_t *tv = vdata + tile_v0;
            const F *tf = vflags + tile_v0;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                unsigned int e[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const unsigned int li = li0 + 4 * u4_off(i) + c;
                    const bool in = li >= lo && li < hi;
                    e[c] = in ? tv[li] : 0u;
                    if (in && tf[li] != 0) hb |= 1u << (4 * i + c);
                }
                x[i] = make_uint4(e[0], e[1], e[2], e[3]);
            }
        }
        // index 0 of the array always opens a segment
        if (tile_v0 <= head && head < tile_v0 + TILE) {
            const unsigned int li = (unsigned int)(head - tile_v0);
            // element li: warp li / CHUNK; within the warp's run, round
            // rem / (32 E), lane (rem % (32 E)) / E, lane-local rem % E
            const unsigned int rem = li % CHUNK, rr = rem / (32u * E), in_r = rem % (32u * E);
            if (li / CHUNK == (unsigned int)warp && in_r / E == (unsigned int)lane) hb |= 1u << (E * rr + in_r % E);
        }
        // Per-round segmented scan within the warp, carry from round to round.
        unsigned int carry = 0;
        pfirst = kNoHead;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned int b = (hb >> (E * r)) & kEMask;
            // the lane's own E elements, scanned with resets at its heads
            unsigned int e[E];
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const unsigned int v = comp(x[Q * r + i / 4], i % 4);
                e[i] = (i == 0 || ((b >> i) & 1u)) ? v : e[i - 1] + v;
            }
            // The round's segmented scan across lanes with a zero carry; every
            // shuffle works on carry-free values, so the rounds overlap and
            // the carry enters by plain arithmetic: a lane gets it when no
            // head lies at or before it in the round.
            const unsigned int t = e[E - 1];
            const unsigned int P = warp_inclusive_sum(t, lane);
            const unsigned int hm = __ballot_sync(0xffffffffu, b != 0u);
            const unsigned int mle = hm & lanemask_le(lane);
            const unsigned int bL = __shfl_sync(0xffffffffu, P - t, 31 - __clz(mle | 1u));
            const unsigned int sl0 = mle ? P - bL : P;
            const unsigned int T0 = __shfl_sync(0xffffffffu, sl0, 31);
            const unsigned int up = __shfl_up_sync(0xffffffffu, sl0, 1);
            const unsigned int cin = lane == 0 ? carry : up + ((hm & lanemask_lt(lane)) == 0u ? carry : 0u);
            if constexpr (WRITE_SCAN) {
#pragma unroll
                for (int i = 0; i < E; ++i)
                    set_comp(x[Q * r + i / 4], i % 4, (b & ((2u << i) - 1u)) ? e[i] : cin + e[i]);
            } else {
                // the reduce needs values at segment ends only: keep the
                // lane-local ones and the lane's carry, added at the ends
#pragma unroll
                for (int i = 0; i < E; ++i) set_comp(x[Q * r + i / 4], i % 4, e[i]);
                cl[r] = cin;
            }
            carry = hm ? T0 : carry + T0;
            if (pfirst == kNoHead && hm) {
                const int lf = __ffs(hm) - 1;
                const unsigned int bf = __shfl_sync(0xffffffffu, b, lf);
                pfirst = 32u * E * r + E * (unsigned int)lf + (unsigned int)(__ffs(bf) - 1);
            }
        }
        const unsigned int wcnt = __reduce_add_sync(0xffffffffu, (unsigned int)__popc(hb));
        if (lane == 0) {
            const int slot = (int)(u & 1u);
            s_wval[slot][warp] = carry;
            s_wcnt[slot][warp] = wcnt;
            s_whas[slot][warp] = pfirst != kNoHead;
            s_wfirst[u % 3][warp] = hb & 1u;
        }
        return t;
    };

    // Store the current tile (first-head slot cs): add each warp's carry-in to the
    // elements before its first head, write the scan, and write each
    // segment's sum at the segment's last element.
    auto store_tile = [&](unsigned int t, int cs, const uint4 (&x)[V], unsigned int hb, unsigned int pfirst,
                          const unsigned int (&cl)[R]) {
        const unsigned long long tile_v0 = (unsigned long long)t * TILE;
        const unsigned int cin = s_bval[warp];
        const bool full = tile_full(t);
        unsigned int lo = 0, hi = TILE;
        if (!full) tile_range(t, lo, hi);
        uint32_t *tv = vdata + tile_v0;
        unsigned int hbase = 0, next_first = 0;
        if (WANT_SUMS) {
            hbase = s_bcnt[warp];
            next_first = warp + 1 < WARPS ? s_wfirst[cs][warp + 1] : s_nexthead;
        }
        // tile-local index of the array's last element (TILE when outside)
        const unsigned long long last_v = head + n - 1 - tile_v0;
        const unsigned int last_li = last_v < TILE ? (unsigned int)last_v : TILE;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned int p0 = 32u * E * r + E * lane;  // warp-local index of the lane's first element
            const unsigned int l0 = li0 + 32u * E * r;        // its tile-local index
            // the scanned value of element i: for the reduce, the lane-local
            // value plus the lane's carry before its first head (computed only
            // where a sum is written)
            auto yv = [&](int i) -> unsigned int {
                unsigned int v = comp(x[Q * r + i / 4], i % 4) + (p0 + i < pfirst ? cin : 0u);
                if constexpr (!WRITE_SCAN)
                    if ((((hb >> (E * r)) & kEMask) & ((2u << i) - 1u)) == 0u) v += cl[r];
                return v;
            };
            unsigned int y[E];
            if constexpr (WRITE_SCAN) {
#pragma unroll
                for (int i = 0; i < E; ++i) y[i] = yv(i);
            }
            if (WRITE_SCAN) {
                if (full) {
#pragma unroll
                    for (int q = 0; q < Q; ++q)
                        __stcs(reinterpret_cast<uint4 *>(tv + l0 + 4 * q),
                               make_uint4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]));
                } else {
#pragma unroll
                    for (int i = 0; i < E; ++i) {
                        const unsigned int li = l0 + i;
                        if (li >= lo && li < hi) tv[li] = y[i];
                    }
                }
            }
            if (WANT_SUMS) {
                const unsigned int b = (hb >> (E * r)) & kEMask;
                // head bit of the element after this lane's last one
                const unsigned int down = __shfl_down_sync(0xffffffffu, b & 1u, 1);
                unsigned int wrap = next_first;
                if (r + 1 < R) wrap = __shfl_sync(0xffffffffu, (hb >> (E * (r + 1))) & 1u, 0);
                const unsigned int after = lane < 31 ? down : wrap;
                // bit i: element i ends a segment (element i + 1 is a head, or
                // element i is the array's last); only elements in the array
                unsigned int ends = (b >> 1) | (after << (E - 1));
                const unsigned int d_last = last_li - l0;
                if (d_last < (unsigned int)E) ends |= 1u << d_last;
                if (!full) {
                    const unsigned int a0 = lo > l0 ? (lo - l0 < (unsigned int)E ? lo - l0 : (unsigned int)E) : 0u;
                    const unsigned int a1 = hi > l0 ? (hi - l0 < (unsigned int)E ? hi - l0 : (unsigned int)E) : 0u;
                    ends &= ((1u << a1) - 1u) & ~((1u << a0) - 1u);
                }
                const unsigned int pc = (unsigned int)__popc(b);
                // Most rounds of long segments hold no segment end: skip them.
                if (__any_sync(0xffffffffu, ends != 0u)) {
                    // sum index of element i's segment: heads before this lane,
                    // plus the lane's heads up to i, minus one (in 64 bits)
                    const unsigned int kb = hbase + (warp_inclusive_sum(pc, lane) - pc);
#pragma unroll
                    for (int i = 0; i < E; ++i) {
                        if ((ends >> i) & 1u) {
                            // at least one head (index 0's) lies at or before every end
                            const unsigned long long k =
                                (unsigned long long)kb + (unsigned int)__popc(b & ((2u << i) - 1u)) - 1ull;
                            if (k < seg_cap) seg_sums[k] = WRITE_SCAN ? y[i] : yv(i);
                        }
                    }
                }
                hbase += __reduce_add_sync(0xffffffffu, pc);
            }
        }
    };

    uint4 xc[V], xn[V];
    unsigned int clc[R], cln[R];  // lanes' carries per round (the reduce only)
    unsigned int hbc = 0, hbn = 0, pfc = kNoHead, pfn = kNoHead;
    unsigned int tc = read_tile(0, xc, hbc, pfc, clc);
    // warp 0 keeps, per lane w < WARPS, what the look-back needs for the
    // current tile: the tile aggregate and warp w's exclusive offsets
    unsigned int agg_val = 0, agg_cnt = 0, wex_val = 0, wex_cnt = 0;
    bool agg_head = false, head_before = false;
    auto block_aggregate = [&](int slot, unsigned int t, unsigned int &a_val, bool &a_head, unsigned int &a_cnt,
                               unsigned int &x_val, bool &h_before, unsigned int &x_cnt) {
        const unsigned int wv = lane < WARPS ? s_wval[slot][lane] : 0u;
        const unsigned int wc = lane < WARPS ? s_wcnt[slot][lane] : 0u;
        const bool wh = lane < WARPS ? s_whas[slot][lane] != 0 : false;
        const unsigned int sw = warp_segmented_inclusive(wv, wh, 0u, lane);
        const unsigned int hm = __ballot_sync(0xffffffffu, wh);
        a_val = __shfl_sync(0xffffffffu, sw, 31);
        a_head = hm != 0;
        const unsigned int cw = warp_inclusive_sum(wc, lane);
        a_cnt = __shfl_sync(0xffffffffu, cw, 31);
        x_val = __shfl_up_sync(0xffffffffu, sw, 1);
        if (lane == 0) x_val = 0;
        h_before = (hm & lanemask_lt(lane)) != 0;
        x_cnt = cw - wc;
        if (lane == 0 && t != skip_tile) {
            // a tile holding a head knows its segmented carry at once
            st_relaxed(desc2 + 2ull * t, tag | (a_head || t == 0 ? (kFlagH | kFlagP) : 0ull) | a_val);
            st_relaxed(desc2 + 2ull * t + 1, tag | (t == 0 ? kFlagP : 0ull) | a_cnt);
        }
    };

    if (!__syncthreads_or(tc >= n_tiles)) {
        if (producer) {
            fence_proxy_async_smem();
            issue(0);
            latest_parity ^= 1u;
        }
        if (warp == 0) block_aggregate(0, tc, agg_val, agg_head, agg_cnt, wex_val, head_before, wex_cnt);
        for (unsigned int u = 1;; ++u) {
            const unsigned int tn = read_tile(u, xn, hbn, pfn, cln);
            const bool more = !__syncthreads_or(tn >= n_tiles);  // barrier A
            unsigned int n_val = 0, n_cnt = 0, n_xval = 0, n_xcnt = 0;
            bool n_head = false, n_before = false;
            if (more && producer) {
                fence_proxy_async_smem();
                const int st = (int)(u % S);
                issue(st);
                latest_parity ^= 1u << st;
            }
            if (warp == 0) {
                if (more) block_aggregate((int)(u & 1u), tn, n_val, n_head, n_cnt, n_xval, n_before, n_xcnt);
                const SegPrefix pre = lookback_seg_wide<U32SCAN_S_LOOKA, U32SCAN_S_LOOKB>(desc2, tc, tag, hdr, limit_ns, lane);
                if (lane == 0 && tc != 0 && tc != skip_tile) {
                    if (!agg_head) st_relaxed(desc2 + 2ull * tc, tag | kFlagP | (unsigned int)(pre.seg + agg_val));
                    st_relaxed(desc2 + 2ull * tc + 1, tag | kFlagP | (unsigned int)(pre.cnt + agg_cnt));
                }
                if (lane < WARPS) {
                    s_bval[lane] = head_before ? wex_val : pre.seg + wex_val;
                    s_bcnt[lane] = pre.cnt + wex_cnt;
                }
                if (lane == 0) {
                    if (tc == n_tiles - 1u && nseg != nullptr) *nseg = pre.cnt + agg_cnt;
                    if (WANT_SUMS) {
                        // head flag of the element just after the tile
                        const unsigned long long after = (unsigned long long)(tc + 1) * TILE;
                        s_nexthead = after < head + n && vflags[after] != 0 ? 1u : 0u;
                    }
                }
            }
            __syncthreads();  // barrier B: carries of the current tile are visible
            store_tile(tc, (int)((u - 1) % 3), xc, hbc, pfc, clc);
            if (!more) break;
#pragma unroll
            for (int r = 0; r < V; ++r) xc[r] = xn[r];
#pragma unroll
            for (int r = 0; r < R; ++r) clc[r] = cln[r];
            hbc = hbn;
            pfc = pfn;
            tc = tn;
            agg_val = n_val;
            agg_head = n_head;
            agg_cnt = n_cnt;
            wex_val = n_xval;
            head_before = n_before;
            wex_cnt = n_xcnt;
        }
    }
    // Leave no bulk copy in flight into this block's shared memory.
    if (producer) {
#pragma unroll
        for (int st = 0; st < S; ++st)
            (void)mbar_wait_bounded(smem_u32(&bar[st]), (latest_parity >> st) & 1u, limit_ns);
    }
}

// Launch shapes, chosen by measurement on GB300 per form and flag type:
// writing the scan favours four elements a lane a round (one u32x4: the
// stores and shared-memory reads stay unit-stride); the reduce, and the scan
// with sums over byte flags, favour eight (half the warp-wide segmented-scan
// work per element). A smaller flag stream leaves room for larger tiles.
// Overridable at build time for tuning sweeps.
#ifndef U32SCAN_S_STAGES
#define U32SCAN_S_STAGES 2
#endif
#ifndef U32SCAN_S_V1
#define U32SCAN_S_V1 7  // u32x4 per lane, four elements a round
#endif
#ifndef U32SCAN_S_V2
#define U32SCAN_S_V2 6  // u32x4 per lane, eight elements a round, int32 flags
#endif
#ifndef U32SCAN_S_V2B
#define U32SCAN_S_V2B 8  // the same with byte flags
#endif
#ifndef U32SCAN_S_T1
#define U32SCAN_S_T1 512  // threads a block, scan only (512 / threads blocks an SM)
#endif
#ifndef U32SCAN_S_T2
#define U32SCAN_S_T2 512  // threads a block, the forms that write sums
#endif
#ifndef U32SCAN_S_STAGES2
#define U32SCAN_S_STAGES2 2  // ring stages of the eight-elements-a-round forms
#endif
template <bool WRITE_SCAN, bool WANT_SUMS, typename F>
constexpr int seg_threads() { return (WRITE_SCAN && !WANT_SUMS) ? U32SCAN_S_T1 : U32SCAN_S_T2; }
template <bool WRITE_SCAN, bool WANT_SUMS, typename F>
constexpr int seg_q() { return (WRITE_SCAN && (!WANT_SUMS || sizeof(F) == 4)) ? 1 : 2; }
template <bool WRITE_SCAN, bool WANT_SUMS, typename F>
constexpr int seg_stages() { return seg_q<WRITE_SCAN, WANT_SUMS, F>() == 1 ? U32SCAN_S_STAGES : U32SCAN_S_STAGES2; }
template <bool WRITE_SCAN, bool WANT_SUMS, typename F>
constexpr int seg_v() {
    return seg_q<WRITE_SCAN, WANT_SUMS, F>() == 1 ? U32SCAN_S_V1 : (sizeof(F) == 1 ? U32SCAN_S_V2B : U32SCAN_S_V2);
}
template <bool WRITE_SCAN, bool WANT_SUMS, typename F>
constexpr unsigned long long seg_tile() {
    return (unsigned long long)seg_threads<WRITE_SCAN, WANT_SUMS, F>() * seg_v<WRITE_SCAN, WANT_SUMS, F>() * 4;
}
template <bool WRITE_SCAN, bool WANT_SUMS, typename F>
constexpr size_t seg_smem() {
    return (size_t)seg_stages<WRITE_SCAN, WANT_SUMS, F>() * seg_tile<WRITE_SCAN, WANT_SUMS, F>() * (4 + sizeof(F));
}
static_assert(seg_smem<true, false, int32_t>() <= 227 * 1024 && seg_smem<true, true, int32_t>() <= 227 * 1024 &&
                  seg_smem<false, true, int32_t>() <= 227 * 1024 && seg_smem<false, true, uint8_t>() <= 227 * 1024 &&
                  seg_smem<true, true, uint8_t>() <= 227 * 1024,
              "shared memory");
// the smallest tile, which has the most tiles, sizes the workspace
constexpr unsigned long long min2(unsigned long long a, unsigned long long b) { return a < b ? a : b; }
constexpr unsigned long long kSTile =
    min2(min2(min2(seg_tile<true, false, int32_t>(), seg_tile<true, true, int32_t>()),
              min2(seg_tile<false, true, int32_t>(), seg_tile<true, false, uint8_t>())),
         min2(seg_tile<true, true, uint8_t>(), seg_tile<false, true, uint8_t>()));

size_t segscan_workspace_bytes(unsigned long long n) {
    const unsigned long long tiles = (n + 3 + kSTile - 1) / kSTile;
    return round_up(kHeaderBytes + 16 * tiles, 256);
}

static std::mutex g_seg_mu;
static int g_seg_sms[64];
static bool g_seg_attr[64][8];

template <bool WRITE_SCAN, bool WANT_SUMS, typename F>
static int segscan_launch(uint32_t *data, const F *flags, unsigned long long n, uint32_t *seg_sums,
                          unsigned long long seg_cap, uint32_t *nseg, void *ws, size_t ws_bytes, cudaStream_t stream,
                          unsigned int skip_tile, unsigned long long limit_ns) {
    if (n >= (1ull << 32)) return U32SCAN_EINVAL;
    if (n > 0 && (data == nullptr || flags == nullptr)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(data) & 3) || (reinterpret_cast<uintptr_t>(flags) & (sizeof(F) - 1)) ||
        (reinterpret_cast<uintptr_t>(seg_sums) & 3) || (reinterpret_cast<uintptr_t>(nseg) & 3))
        return U32SCAN_EINVAL;
    if (n == 0) {
        if (nseg && cudaMemsetAsync(nseg, 0, sizeof(uint32_t), stream) != cudaSuccess) return U32SCAN_ECUDA;
        return U32SCAN_OK;
    }
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < segscan_workspace_bytes(n))
        return U32SCAN_EWORKSPACE;
    const unsigned int head = (unsigned int)((reinterpret_cast<uintptr_t>(data) & 15) >> 2);
    // flags stream by bulk copy when they start a tile on a 16-byte boundary too
    const int aligned = ((reinterpret_cast<uintptr_t>(flags) - sizeof(F) * head) & 15) == 0;
    constexpr unsigned long long TILE = seg_tile<WRITE_SCAN, WANT_SUMS, F>();
    const unsigned int n_tiles = (unsigned int)((n + head + TILE - 1) / TILE);
    constexpr int THREADS = seg_threads<WRITE_SCAN, WANT_SUMS, F>();
    auto kern = segscan_u32_persistent<THREADS, seg_v<WRITE_SCAN, WANT_SUMS, F>(), seg_q<WRITE_SCAN, WANT_SUMS, F>(),
                                       seg_stages<WRITE_SCAN, WANT_SUMS, F>(), WRITE_SCAN, WANT_SUMS, F>;
    constexpr size_t smem = seg_smem<WRITE_SCAN, WANT_SUMS, F>();
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    int sms;
    {
        std::lock_guard<std::mutex> lock(g_seg_mu);
        if (g_seg_sms[dev] == 0 &&
            cudaDeviceGetAttribute(&g_seg_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return U32SCAN_ECUDA;
        const int which = (sizeof(F) == 1 ? 4 : 0) + (WRITE_SCAN ? 2 : 0) + (WANT_SUMS ? 1 : 0);
        if (!g_seg_attr[dev][which]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return U32SCAN_ECUDA;
            g_seg_attr[dev][which] = true;
        }
        sms = g_seg_sms[dev];
    }
    const unsigned int slots = (unsigned int)sms * (512u / THREADS);  // blocks resident at once
    const unsigned int grid = n_tiles < slots ? n_tiles : slots;
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    unsigned long long *desc2 = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kHeaderBytes);
    kern<<<grid, THREADS, smem, stream>>>(data, flags, n, seg_sums, seg_cap, nseg, hdr, desc2, n_tiles, head,
                                             aligned, skip_tile, limit_ns);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int segscan_inclusive_u32(uint32_t *data, const int32_t *head_flags, size_t n, uint32_t *seg_sums,
                                     size_t seg_capacity, uint32_t *nseg, void *ws, size_t ws_bytes,
                                     u32scan_stream_t stream) {
    if (seg_sums != nullptr)
        return segscan_launch<true, true>(data, head_flags, n, seg_sums, seg_capacity, nseg, ws, ws_bytes,
                                          (cudaStream_t)stream, 0xffffffffu, kDefaultLimitNs);
    return segscan_launch<true, false>(data, head_flags, n, nullptr, 0, nseg, ws, ws_bytes, (cudaStream_t)stream,
                                       0xffffffffu, kDefaultLimitNs);
}

extern "C" int segreduce_u32(const uint32_t *data, const int32_t *head_flags, size_t n, uint32_t *seg_sums,
                             size_t seg_capacity, uint32_t *nseg, void *ws, size_t ws_bytes,
                             u32scan_stream_t stream) {
    if (seg_sums == nullptr && nseg == nullptr) return U32SCAN_EINVAL;
    return segscan_launch<false, true>(const_cast<uint32_t *>(data), head_flags, n, seg_sums,
                                       seg_sums ? seg_capacity : 0, nseg, ws, ws_bytes, (cudaStream_t)stream,
                                       0xffffffffu, kDefaultLimitNs);
}

extern "C" int segscan_inclusive_u32_u8heads(uint32_t *data, const uint8_t *head_flags, size_t n, uint32_t *seg_sums,
                                             size_t seg_capacity, uint32_t *nseg, void *ws, size_t ws_bytes,
                                             u32scan_stream_t stream) {
    if (seg_sums != nullptr)
        return segscan_launch<true, true>(data, head_flags, n, seg_sums, seg_capacity, nseg, ws, ws_bytes,
                                          (cudaStream_t)stream, 0xffffffffu, kDefaultLimitNs);
    return segscan_launch<true, false>(data, head_flags, n, nullptr, 0, nseg, ws, ws_bytes, (cudaStream_t)stream,
                                       0xffffffffu, kDefaultLimitNs);
}

extern "C" int segreduce_u32_u8heads(const uint32_t *data, const uint8_t *head_flags, size_t n, uint32_t *seg_sums,
                                     size_t seg_capacity, uint32_t *nseg, void *ws, size_t ws_bytes,
                                     u32scan_stream_t stream) {
    if (seg_sums == nullptr && nseg == nullptr) return U32SCAN_EINVAL;
    return segscan_launch<false, true>(const_cast<uint32_t *>(data), head_flags, n, seg_sums,
                                       seg_sums ? seg_capacity : 0, nseg, ws, ws_bytes, (cudaStream_t)stream,
                                       0xffffffffu, kDefaultLimitNs);
}

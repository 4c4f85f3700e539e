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
// head count gives every segment end its index into the sums. Warp 0 walks
// the value and warp 1 the head count, so the two walks overlap (one warp
// walking both, the value first, measured 3 % slower for the scan with
// sums). The forms without sums need no such index: they walk the value
// alone, and count the segments with one atomic add a tile.
//
// Layout inside a tile (lane runs): lane l of warp w owns the E = 4R
// consecutive elements at w * 32E + l * E of the tile (R u32x4, R odd: a
// warp reading its lanes' i-th u32x4 from the linear shared-memory stage then
// hits eight different 16-byte bank groups in every quarter-warp, so the
// reads are free of bank conflicts). Head flags become one bit per element
// (bit j: element j of the run); byte flags are read four to a word and
// tested bytewise. A lane scans its run sequentially with resets at its
// heads; one warp-wide segmented scan of the lanes' run values then serves
// E elements a lane, and a lane's segment ends take consecutive indices into
// the sums. The forms that write the scan put it in a shared-memory output
// buffer (the same layout, conflict free) and store each full tile with one
// 1-D bulk copy.
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
#ifndef U32SCAN_S_STAGEMIN
#define U32SCAN_S_STAGEMIN 64  // fewest ends a warp for which its sums are staged
#endif
#ifndef U32SCAN_S_FEWENDS
#define U32SCAN_S_FEWENDS 2  // segment ends a lane up to which its sums are visited end by end (no buffer)
#endif
#ifndef U32SCAN_S_ATOMCOUNT
#define U32SCAN_S_ATOMCOUNT 1  // without sums: the segment count by one atomic add a tile, no count look-back
#endif

namespace u32scan {

// The segment count of the forms without sums, which need no segment index
// per tile: every tile adds 2^32 + (its head count) to one 64-bit word of
// the workspace header (a spare word no other kernel uses, at byte 128, away
// from the 128-byte line of the tile counter). The add that finds
// n_tiles - 1 tiles counted before it is the last, so its old value plus
// its own count is the total; that tile puts the word back to zero for the
// next call. The heads of a whole array number fewer than 2^32, so they
// never carry into the tile count. (A compare-and-swap loop on a word in
// the tile counter's line measured 13 times slower than the look-back.)
__device__ __forceinline__ unsigned long long *seg_count_word(WsHeader *hdr) { return &hdr->seg_count; }

__device__ __forceinline__ bool seg_count_add(WsHeader *hdr, unsigned int n_tiles, unsigned int heads,
                                              unsigned int &total) {
    unsigned long long *w = seg_count_word(hdr);
    const unsigned long long old = atomicAdd(w, (1ull << 32) | (unsigned long long)heads);
    if ((unsigned int)(old >> 32) != n_tiles - 1u) return false;
    total = (unsigned int)old + heads;
    atomicExch(w, 0ull);
    return true;
}

// Element j (0 <= j < 4R, known only at run time) of a run held in
// registers, by predicated moves: the u32x4 first, then the component.
template <int R>
__device__ __forceinline__ unsigned int pick(const uint4 (&x)[R], unsigned int j) {
    // bitwise blends under an all-ones / all-zeros mask, so that the run stays
    // in registers (no indexed copy in local memory)
    const unsigned int qi = j >> 2;
    uint4 q = x[0];
#pragma unroll
    for (int i = 1; i < R; ++i) {
        const unsigned int m = 0u - (unsigned int)(qi == (unsigned int)i);
        q.x = (x[i].x & m) | (q.x & ~m);
        q.y = (x[i].y & m) | (q.y & ~m);
        q.z = (x[i].z & m) | (q.z & ~m);
        q.w = (x[i].w & m) | (q.w & ~m);
    }
    const unsigned int c = j & 3u;
    const unsigned int lo = (c & 1u) ? q.y : q.x, hi = (c & 1u) ? q.w : q.z;
    return (c & 2u) ? hi : lo;
}

// Component c of a u32x4.
__device__ __forceinline__ unsigned int comp(const uint4 &v, int c) {
    return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}
__device__ __forceinline__ void set_comp(uint4 &v, int c, unsigned int a) {
    if (c == 0) v.x = a; else if (c == 1) v.y = a; else if (c == 2) v.z = a; else v.w = a;
}

// The kernel: persistent, one 512-thread block per SM; tile layout, pipeline
// and look-back as described at the top of this file.
template <int THREADS, int R, int S, bool WRITE_SCAN, bool WANT_SUMS, typename F, bool BUF, int SUMCAP>
__global__ void __launch_bounds__(THREADS, 512 / THREADS)
segscan_lanes_persistent(uint32_t *__restrict__ data, const F *__restrict__ flags, unsigned long long n,
                         uint32_t *seg_sums, unsigned long long seg_cap, uint32_t *nseg, WsHeader *hdr,
                         unsigned long long *desc2, unsigned int n_tiles, unsigned int head, int streams_aligned,
                         unsigned int skip_tile, unsigned long long limit_ns, unsigned long long clear_words) {
    constexpr int WARPS = THREADS / 32;
    constexpr bool ATOM_COUNT = !WANT_SUMS && U32SCAN_S_ATOMCOUNT;  // the count serves no segment index
    constexpr int E = 4 * R;                    // elements a lane
    constexpr unsigned int CHUNK = 32u * E;     // elements a warp
    constexpr unsigned int TILE = WARPS * CHUNK;
    constexpr unsigned int TILE_BYTES = TILE * 4;
    constexpr unsigned int FLAG_BYTES = TILE * (unsigned int)sizeof(F);
    constexpr unsigned int STAGE_U4 = (TILE_BYTES + FLAG_BYTES) / 16;
    static_assert(R % 2 == 1 && E <= 32, "odd u32x4 count a lane; a lane's head bits fit a word");
    static_assert(WARPS <= 32 && FLAG_BYTES % 16 == 0, "one lane per warp; whole 16-byte flag stages");
    static_assert(sizeof(F) == 4 || sizeof(F) == 1, "int32 or byte head flags");
    // BUF: a tile-sized shared-memory buffer after the stages, in the lane-run
    // layout. The forms writing the scan put the tile's scan there and store
    // it with one bulk copy; the reduce keeps each lane's scanned run in its
    // own part of it, to read the values at segment ends by index.
    extern __shared__ __align__(128) uint4 stage_buf[];  // S stages of [values | flags] (+ the buffer)
    __shared__ __align__(8) unsigned long long bar[S];
    __shared__ unsigned int s_tile[S];
    __shared__ unsigned int s_wval[2][WARPS], s_wcnt[2][WARPS], s_whas[2][WARPS];
    __shared__ unsigned int s_wfirst[3][WARPS];  // head bit of each warp's first element, three tiles deep
    __shared__ unsigned int s_bval[WARPS], s_bcnt[WARPS], s_nexthead;
    __shared__ unsigned int s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned int last_draw = n_tiles + (unsigned int)S * gridDim.x - 1u;
    uint32_t *vdata = reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(data) - 4ull * head);
    const F *vflags = reinterpret_cast<const F *>(reinterpret_cast<uintptr_t>(flags) - sizeof(F) * head);
    const bool producer = threadIdx.x == THREADS - 32;
    unsigned int latest_parity = 0;
    const unsigned int li0 = (unsigned int)warp * CHUNK + (unsigned int)E * (unsigned int)lane;  // lane's first element

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
    volatile unsigned int *vs_tile = s_tile;

    // What a lane keeps of a tile between reading it and storing it.
    struct LaneRun {
        uint4 x[R];           // the run, then its segmented scan from the lane's start
        unsigned int hb;      // head bits (bit j: element j of the run)
        unsigned int cin;     // segmented value flowing in from the warp's earlier lanes
        unsigned int cex;     // heads in the warp's earlier lanes (the forms with sums)
        bool head_before;     // a head in the warp's earlier lanes
    };

    // Read draw u (stage u % S) into a lane run, scan it, and leave the warp
    // aggregates in slot u & 1. Returns the tile, n_tiles past the end, or
    // n_tiles + 1 on a timeout.
    auto read_tile = [&](unsigned int u, LaneRun &L) -> unsigned int {
        const int st = (int)(u % S);
        if (!mbar_wait_bounded(smem_u32(&bar[st]), (u / S) & 1u, limit_ns)) {
            report_timeout(hdr, 0xfffffffeu);
            return n_tiles + 1u;
        }
        const unsigned int t = vs_tile[st];
        if (t >= n_tiles) return n_tiles;
        const unsigned long long tile_v0 = (unsigned long long)t * TILE;
        unsigned int hb = 0;
        if (tile_full(t)) {
            const uint4 *sv = stage_buf + st * STAGE_U4 + (li0 >> 2);
            if constexpr (sizeof(F) == 4) {
                const int4 *sf = reinterpret_cast<const int4 *>(stage_buf + st * STAGE_U4 + TILE / 4) + (li0 >> 2);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    L.x[i] = sv[i];
                    const int4 f = sf[i];
                    hb |= ((f.x != 0) | ((f.y != 0) << 1) | ((f.z != 0) << 2) | ((f.w != 0) << 3)) << (4 * i);
                }
            } else {
                // four byte flags in one word: byte c non-zero -> bit c of a nibble
                const unsigned int *sf =
                    reinterpret_cast<const unsigned int *>(stage_buf + st * STAGE_U4 + TILE / 4) + (li0 >> 2);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    L.x[i] = sv[i];
                    const unsigned int m = __vcmpne4(sf[i], 0u) & 0x08040201u;
                    hb |= ((m * 0x01010101u) >> 24) << (4 * i);
                }
            }
        } else {
            unsigned int lo, hi;
            tile_range(t, lo, hi);
            const uint32_t *tv = vdata + tile_v0;
            const F *tf = vflags + tile_v0;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                unsigned int e[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const unsigned int li = li0 + 4 * i + c;
                    const bool in = li >= lo && li < hi;
                    e[c] = in ? tv[li] : 0u;
                    if (in && tf[li] != 0) hb |= 1u << (4 * i + c);
                }
                L.x[i] = make_uint4(e[0], e[1], e[2], e[3]);
            }
        }
        // index 0 of the array always opens a segment
        if (tile_v0 <= head && head < tile_v0 + TILE) {
            const unsigned int li = (unsigned int)(head - tile_v0);
            if (li - li0 < (unsigned int)E) hb |= 1u << (li - li0);
        }
        // the lane's run, scanned with resets at its heads
        unsigned int s = 0;
#pragma unroll
        for (int j = 0; j < E; ++j) {
            const unsigned int v = comp(L.x[j / 4], j % 4);
            s = ((hb >> j) & 1u) ? v : s + v;
            set_comp(L.x[j / 4], j % 4, s);
        }
        // across the warp's lanes: the value at the end of lane l's run with
        // no carry into the warp is P[l] - P[L-1], L the last lane at or
        // before l holding a head (P[l] when there is none)
        const unsigned int P = warp_inclusive_sum(s, lane);
        const unsigned int hm = __ballot_sync(0xffffffffu, hb != 0u);
        const unsigned int mle = hm & lanemask_le(lane);
        const unsigned int bL = __shfl_sync(0xffffffffu, P - s, 31 - __clz(mle | 1u));
        const unsigned int incl = mle ? P - bL : P;
        const unsigned int up = __shfl_up_sync(0xffffffffu, incl, 1);
        L.cin = lane == 0 ? 0u : up;
        L.head_before = (hm & lanemask_lt(lane)) != 0u;
        L.hb = hb;
        const unsigned int pc = (unsigned int)__popc(hb);
        L.cex = WANT_SUMS ? warp_inclusive_sum(pc, lane) - pc : 0u;
        const unsigned int wcnt = __reduce_add_sync(0xffffffffu, pc);
        if (lane == 31) {
            const int slot = (int)(u & 1u);
            s_wval[slot][warp] = incl;
            s_wcnt[slot][warp] = wcnt;
            s_whas[slot][warp] = hm != 0u;
        }
        if (lane == 0) s_wfirst[u % 3][warp] = hb & 1u;
        return t;
    };

    // Store the current tile (first-head slot cs): each lane adds its carry
    // to the elements before its first head, writes the scan, and writes the
    // sum of each segment that ends in its run.
    auto store_tile = [&](unsigned int t, int cs, const LaneRun &L) {
        const unsigned long long tile_v0 = (unsigned long long)t * TILE;
        const bool full = tile_full(t);
        unsigned int lo = 0, hi = TILE;
        if (!full) tile_range(t, lo, hi);
        uint32_t *tv = vdata + tile_v0;
        const unsigned int wc = s_bval[warp];
        const unsigned int lc = L.head_before ? L.cin : wc + L.cin;  // flows into the lane's run
        const unsigned int f = L.hb ? (unsigned int)(__ffs(L.hb) - 1) : (unsigned int)E;  // first head
        auto y = [&](int j) -> unsigned int { return comp(L.x[j / 4], j % 4) + ((unsigned int)j < f ? lc : 0u); };
        uint4 *ob = stage_buf + S * STAGE_U4 + (li0 >> 2);  // this lane's run in the buffer (BUF)
        if (WRITE_SCAN) {
            if (full && BUF) {
                // through the output buffer (same lane-run layout, conflict
                // free), then one 1-D bulk copy of the whole tile; thread 0
                // waited for its previous copy to read the buffer before
                // barrier B, and tile_full(t) is the same for every thread
#pragma unroll
                for (int i = 0; i < R; ++i) ob[i] = make_uint4(y(4 * i), y(4 * i + 1), y(4 * i + 2), y(4 * i + 3));
                fence_proxy_async_smem();
                __syncthreads();  // barrier C: the output buffer is complete
                if (threadIdx.x == 0) bulk_store(tv, smem_u32(stage_buf + S * STAGE_U4), TILE_BYTES);
            } else if (full) {
#pragma unroll
                for (int i = 0; i < R; ++i)
                    *reinterpret_cast<uint4 *>(tv + li0 + 4 * i) = make_uint4(y(4 * i), y(4 * i + 1), y(4 * i + 2), y(4 * i + 3));
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    const unsigned int li = li0 + j;
                    if (li >= lo && li < hi) tv[li] = y(j);
                }
            }
        }
        if (WANT_SUMS) {
            // element j ends a segment when element j + 1 is a head (the next
            // lane's, warp's or tile's first element after the run's last) or
            // j is the array's last element; only elements in the array count
            const unsigned int down = __shfl_down_sync(0xffffffffu, L.hb & 1u, 1);
            const unsigned int next_first = warp + 1 < WARPS ? s_wfirst[cs][warp + 1] : s_nexthead;
            const unsigned int after = lane < 31 ? down : next_first;
            unsigned int ends = (L.hb >> 1) | (after << (E - 1));
            const unsigned long long last_v = head + n - 1 - tile_v0;
            const unsigned int last_li = last_v < TILE ? (unsigned int)last_v : TILE;
            const unsigned int d_last = last_li - li0;
            if (d_last < (unsigned int)E) ends |= 1u << d_last;
            if (!full) {
                const unsigned int a0 = lo > li0 ? (lo - li0 < (unsigned int)E ? lo - li0 : (unsigned int)E) : 0u;
                const unsigned int a1 = hi > li0 ? (hi - li0 < (unsigned int)E ? hi - li0 : (unsigned int)E) : 0u;
                ends &= (unsigned int)(((1ull << a1) - 1ull) & ~((1ull << a0) - 1ull));
            }
            ends &= (unsigned int)((1ull << E) - 1ull);
            // segment index of element j: the heads before the run plus those
            // of the run up to j, minus one (index 0's head lies at or before
            // every end)
            const unsigned int k0 = s_bcnt[warp] + L.cex - 1u;
            // A warp's ends take consecutive segment indices (one head lies
            // between two ends), so a warp with at most SUMCAP ends in a full
            // tile puts its sums in its own shared-memory slots (the m-th end
            // of a lane at the lane's exclusive end count + m) and writes them
            // with unit-stride stores; otherwise each lane stores its own.
            bool staged = false;
            unsigned int ecx = 0, cw = 0, kw = 0;
            uint32_t *stg = nullptr;
            if constexpr (SUMCAP > 0) {
                if (full) {
                    const unsigned int ne = (unsigned int)__popc(ends);
                    cw = __reduce_add_sync(0xffffffffu, ne);
                    // the same for the whole warp; few ends go straight out
                    staged = cw >= U32SCAN_S_STAGEMIN && cw <= (unsigned int)SUMCAP;
                    if (staged) {
                        ecx = warp_inclusive_sum(ne, lane) - ne;
                        // the warp's first end: its lowest lane with ends, that lane's first
                        const unsigned int hmE = __ballot_sync(0xffffffffu, ne != 0u);
                        const unsigned int j0 = ends ? (unsigned int)(__ffs(ends) - 1) : 0u;
                        const unsigned int kf = k0 + (unsigned int)__popc(L.hb & ((2u << j0) - 1u));
                        kw = __shfl_sync(0xffffffffu, kf, hmE ? __ffs(hmE) - 1 : 0);
                        stg = reinterpret_cast<uint32_t *>(stage_buf + S * STAGE_U4 + (BUF ? TILE / 4 : 0)) +
                              (unsigned int)warp * SUMCAP;
                    }
                }
            }
            // the m-th end of this lane, in segment k, with value v
            auto emit = [&](unsigned int m, unsigned int k, unsigned int v) {
                if (staged)
                    stg[ecx + m] = v;
                else if ((unsigned long long)k < seg_cap)
                    seg_sums[k] = v;
            };
            if (BUF && full) {
                // the run's scan is in the buffer (the forms writing the scan
                // put it there above; the reduce writes it now, into this
                // lane's own part): visit the ends only
                if (!WRITE_SCAN && ends != 0u) {
#pragma unroll
                    for (int i = 0; i < R; ++i) ob[i] = make_uint4(y(4 * i), y(4 * i + 1), y(4 * i + 2), y(4 * i + 3));
                }
                const uint32_t *run = reinterpret_cast<const uint32_t *>(ob);
                unsigned int m = 0;
                for (unsigned int e = ends; e != 0u; e &= e - 1u, ++m) {
                    const unsigned int j = (unsigned int)(__ffs(e) - 1);
                    emit(m, staged ? 0u : k0 + (unsigned int)__popc(L.hb & ((2u << j) - 1u)), run[j]);
                }
            } else if (__any_sync(0xffffffffu, __popc(ends) > U32SCAN_S_FEWENDS)) {
                // many ends in some lane: one pass over the run's elements
                unsigned int k = k0, m = 0;
#pragma unroll
                for (int j = 0; j < E; ++j) {
                    k += (L.hb >> j) & 1u;
                    if ((ends >> j) & 1u) emit(m++, k, y(j));
                }
            } else {
                // few ends a lane: visit them, picking each value out of the registers
                unsigned int m = 0;
                for (unsigned int e = ends; e != 0u; e &= e - 1u, ++m) {
                    const unsigned int j = (unsigned int)(__ffs(e) - 1);
                    emit(m, staged ? 0u : k0 + (unsigned int)__popc(L.hb & ((2u << j) - 1u)),
                         pick<R>(L.x, j) + (j < f ? lc : 0u));
                }
            }
            if (staged) {
                __syncwarp();
                for (unsigned int i = (unsigned int)lane; i < cw; i += 32u)
                    if ((unsigned long long)(kw + i) < seg_cap) seg_sums[kw + i] = stg[i];
                __syncwarp();
            }
        }
    };

    // Head flag of the element just after tile t (warp 0, lane 0, the forms
    // with sums): loaded one round before it is needed, when the tile is
    // read, so that its latency stays off the look-back's path.
    auto head_after = [&](unsigned int t) -> unsigned int {
        const unsigned long long after = (unsigned long long)(t + 1) * TILE;
        return after < head + n && vflags[after] != 0 ? 1u : 0u;
    };
    LaneRun Lc, Ln;
    unsigned int tc = read_tile(0, Lc);
    unsigned int nh_c = 0, nh_n = 0;
    if (WANT_SUMS && threadIdx.x == 0 && tc < n_tiles) nh_c = head_after(tc);
    // The walking warps keep, per lane w < WARPS, what the look-back needs
    // for the current tile: the tile aggregate and warp w's exclusive
    // offsets (warp 0 the value's, the count's warp the head count's).
    unsigned int agg_val = 0, agg_cnt = 0, wex_val = 0, wex_cnt = 0;
    bool agg_head = false, head_before = false;
    // Both aggregates in warp 0 (the forms counting segments by atomic add).
    auto block_aggregate = [&](int slot, unsigned int t, unsigned int &a_val, bool &a_head, unsigned int &a_cnt,
                               unsigned int &x_val, bool &h_before, unsigned int &x_cnt) {
        const unsigned int wv = lane < WARPS ? s_wval[slot][lane] : 0u;
        const unsigned int wcn = lane < WARPS ? s_wcnt[slot][lane] : 0u;
        const bool wh = lane < WARPS ? s_whas[slot][lane] != 0 : false;
        const unsigned int sw = warp_segmented_inclusive(wv, wh, 0u, lane);
        const unsigned int hm = __ballot_sync(0xffffffffu, wh);
        a_val = __shfl_sync(0xffffffffu, sw, 31);
        a_head = hm != 0;
        const unsigned int cw = warp_inclusive_sum(wcn, lane);
        a_cnt = __shfl_sync(0xffffffffu, cw, 31);
        x_val = __shfl_up_sync(0xffffffffu, sw, 1);
        if (lane == 0) x_val = 0;
        h_before = (hm & lanemask_lt(lane)) != 0;
        x_cnt = cw - wcn;
        if (lane == 0 && t != skip_tile)  // a tile holding a head knows its segmented carry at once
            st_relaxed(desc2 + 2ull * t, tag | (a_head || t == 0 ? (kFlagH | kFlagP) : 0ull) | a_val);
    };
    // With a walked head count (the forms with sums), warp 0 takes the
    // segmented value and warp 1 the head count, each its own aggregate and
    // look-back, so that the two walks overlap.
    auto value_aggregate = [&](int slot, unsigned int t, unsigned int &a_val, bool &a_head, unsigned int &x_val,
                               bool &h_before) {
        const unsigned int wv = lane < WARPS ? s_wval[slot][lane] : 0u;
        const bool wh = lane < WARPS ? s_whas[slot][lane] != 0 : false;
        const unsigned int sw = warp_segmented_inclusive(wv, wh, 0u, lane);
        const unsigned int hm = __ballot_sync(0xffffffffu, wh);
        a_val = __shfl_sync(0xffffffffu, sw, 31);
        a_head = hm != 0;
        x_val = __shfl_up_sync(0xffffffffu, sw, 1);
        if (lane == 0) x_val = 0;
        h_before = (hm & lanemask_lt(lane)) != 0;
        if (lane == 0 && t != skip_tile)
            st_relaxed(desc2 + 2ull * t, tag | (a_head || t == 0 ? (kFlagH | kFlagP) : 0ull) | a_val);
    };
    auto count_aggregate = [&](int slot, unsigned int t, unsigned int &a_cnt, unsigned int &x_cnt) {
        const unsigned int wcn = lane < WARPS ? s_wcnt[slot][lane] : 0u;
        const unsigned int cw = warp_inclusive_sum(wcn, lane);
        a_cnt = __shfl_sync(0xffffffffu, cw, 31);
        x_cnt = cw - wcn;
        if (lane == 0 && t != skip_tile) st_relaxed(desc2 + 2ull * t + 1, tag | (t == 0 ? kFlagP : 0ull) | a_cnt);
    };

    if (!__syncthreads_or(tc >= n_tiles)) {
        if (producer) {
            fence_proxy_async_smem();
            issue(0);
            latest_parity ^= 1u;
        }
        if constexpr (ATOM_COUNT) {
            if (warp == 0) block_aggregate(0, tc, agg_val, agg_head, agg_cnt, wex_val, head_before, wex_cnt);
        } else {
            if (warp == 0) value_aggregate(0, tc, agg_val, agg_head, wex_val, head_before);
            if (warp == 1) count_aggregate(0, tc, agg_cnt, wex_cnt);
        }
        for (unsigned int u = 1;; ++u) {
            const unsigned int tn = read_tile(u, Ln);
            const bool more = !__syncthreads_or(tn >= n_tiles);  // barrier A
            if (WANT_SUMS && threadIdx.x == 0 && more) nh_n = head_after(tn);
            unsigned int n_val = 0, n_cnt = 0, n_xval = 0, n_xcnt = 0;
            bool n_head = false, n_before = false;
            if (more && producer) {
                fence_proxy_async_smem();
                const int st = (int)(u % S);
                issue(st);
                latest_parity ^= 1u << st;
            }
            if (!ATOM_COUNT && warp == 0) {
                // the segmented value, walked while warp 1 walks the head count;
                // its first window is loaded before the next tile's aggregate
                unsigned long long wa[U32SCAN_S_LOOKA];
                if (tc != 0) lookback_window<U32SCAN_S_LOOKA, kAdd, 2>(desc2, (long long)tc - 1, tag, lane, wa);
                if (more) value_aggregate((int)(u & 1u), tn, n_val, n_head, n_xval, n_before);
                unsigned int seg = 0;
                if (tc != 0) {
                    seg = lookback_prefix_wide<U32SCAN_S_LOOKA, kAdd, 2, kFlagP | kFlagH>(desc2, tc, tag, hdr,
                                                                                        limit_ns, lane, wa);
                }
                if (lane == 0 && tc != 0 && tc != skip_tile && !agg_head)
                    st_relaxed(desc2 + 2ull * tc, tag | kFlagP | (unsigned int)(seg + agg_val));
                if (lane < WARPS) s_bval[lane] = head_before ? wex_val : seg + wex_val;
                if (WANT_SUMS && lane == 0) s_nexthead = nh_c;
            } else if (!ATOM_COUNT && warp == 1) {
                unsigned long long wb[U32SCAN_S_LOOKB];
                if (tc != 0) lookback_window<U32SCAN_S_LOOKB, kAdd, 2>(desc2 + 1, (long long)tc - 1, tag, lane, wb);
                if (more) count_aggregate((int)(u & 1u), tn, n_cnt, n_xcnt);
                unsigned int cnt = 0;
                if (tc != 0) {
                    cnt = lookback_prefix_wide<U32SCAN_S_LOOKB, kAdd, 2, kFlagP>(desc2 + 1, tc, tag, hdr, limit_ns,
                                                                                 lane, wb);
                }
                if (lane == 0 && tc != 0 && tc != skip_tile)
                    st_relaxed(desc2 + 2ull * tc + 1, tag | kFlagP | (unsigned int)(cnt + agg_cnt));
                if (lane < WARPS) s_bcnt[lane] = cnt + wex_cnt;
                if (lane == 0 && tc == n_tiles - 1u && nseg != nullptr) *nseg = cnt + agg_cnt;
            } else if (ATOM_COUNT && warp == 0) {
                // the value alone; the segments are counted by one atomic add
                unsigned long long wa[U32SCAN_S_LOOKA];
                if (tc != 0) lookback_window<U32SCAN_S_LOOKA, kAdd, 2>(desc2, (long long)tc - 1, tag, lane, wa);
                if (more) block_aggregate((int)(u & 1u), tn, n_val, n_head, n_cnt, n_xval, n_before, n_xcnt);
                unsigned int seg = 0;
                if (tc != 0) {
                    seg = lookback_prefix_wide<U32SCAN_S_LOOKA, kAdd, 2, kFlagP | kFlagH>(desc2, tc, tag, hdr,
                                                                                        limit_ns, lane, wa);
                }
                if (lane == 0 && tc != 0 && tc != skip_tile && !agg_head)
                    st_relaxed(desc2 + 2ull * tc, tag | kFlagP | (unsigned int)(seg + agg_val));
                if (lane < WARPS) s_bval[lane] = head_before ? wex_val : seg + wex_val;
                if (lane == 0) {
                    unsigned int total;
                    if (nseg != nullptr && seg_count_add(hdr, n_tiles, agg_cnt, total)) *nseg = total;
                    if (WANT_SUMS) s_nexthead = nh_c;
                }
            }
            if (WRITE_SCAN && BUF && threadIdx.x == 0) bulk_wait_read();  // output buffer free again
            __syncthreads();  // barrier B: carries of the current tile are visible
            store_tile(tc, (int)((u - 1) % 3), Lc);
            if (!more) break;
            Lc = Ln;
            tc = tn;
            nh_c = nh_n;
            agg_val = n_val;
            agg_head = n_head;
            agg_cnt = n_cnt;
            wex_val = n_xval;
            head_before = n_before;
            wex_cnt = n_xcnt;
        }
    }
    // Leave no bulk copy in flight into or out of this block's shared memory.
    if (producer) {
#pragma unroll
        for (int st = 0; st < S; ++st)
            (void)mbar_wait_bounded(smem_u32(&bar[st]), (latest_parity >> st) & 1u, limit_ns);
    }
    if (WRITE_SCAN && BUF && threadIdx.x == 0) bulk_wait_all();
    finish_period(hdr, s_epoch, desc2, clear_words);
}

// Launch shapes, chosen by measurement on GB300 (n = 2^26) and overridable
// at build time for tuning sweeps: R u32x4 a lane (odd), ring stages, and
// whether the forms that write the scan go through an output buffer and a
// bulk copy. Writing the scan from registers (each lane's 16-byte stores
// fill half a 32-byte sector: twice the store requests of unit-stride
// stores) measured slower than the buffer; the buffer leaves room for R = 5
// with int32 flags and R = 7 with byte flags.
#ifndef U32SCAN_S_LR
#define U32SCAN_S_LR 7  // the reduce: u32x4 a lane
#endif
#ifndef U32SCAN_S_LSTAGES4
#define U32SCAN_S_LSTAGES4 2  // the reduce: ring stages with int32 flags
#endif
#ifndef U32SCAN_S_LSTAGES1
#define U32SCAN_S_LSTAGES1 3  // and with byte flags
#endif
#ifndef U32SCAN_S_WOUT
#define U32SCAN_S_WOUT 1  // the forms writing the scan: through an output buffer and a bulk copy
#endif
// The reduce with the runs kept in a shared-memory buffer (and the shapes of
// the forms writing the scan), per flag type; without it, a lane with few
// segment ends picks their values out of its registers. Measured (Gelem/s,
// geometric / length-4 heads): int32 flags 472 / 396 with the buffer (R = 5)
// against 588 / 449 without (R = 7, larger tiles); byte flags 620 / 456
// against 631 / 475.
#ifndef U32SCAN_S_RBUF4
#define U32SCAN_S_RBUF4 0
#endif
#ifndef U32SCAN_S_RBUF1
#define U32SCAN_S_RBUF1 0
#endif
#ifndef U32SCAN_S_WR4
#define U32SCAN_S_WR4 5  // the forms writing the scan: u32x4 a lane with int32 flags
#endif
#ifndef U32SCAN_S_WR1
#define U32SCAN_S_WR1 7  // and with byte flags
#endif
template <bool WRITE_SCAN, typename F>
constexpr bool lanes_out() { return WRITE_SCAN ? U32SCAN_S_WOUT : sizeof(F) == 1 ? U32SCAN_S_RBUF1 : U32SCAN_S_RBUF4; }
template <bool WRITE_SCAN, typename F>
constexpr int lanes_r() { return !lanes_out<WRITE_SCAN, F>() ? U32SCAN_S_LR : sizeof(F) == 1 ? U32SCAN_S_WR1 : U32SCAN_S_WR4; }
template <bool WRITE_SCAN, typename F>
constexpr int lanes_stages() {
    return lanes_out<WRITE_SCAN, F>() ? 2 : sizeof(F) == 1 ? U32SCAN_S_LSTAGES1 : U32SCAN_S_LSTAGES4;
}
template <bool WRITE_SCAN, typename F>
constexpr unsigned long long lanes_tile() { return 512ull * 4 * lanes_r<WRITE_SCAN, F>(); }
template <bool WRITE_SCAN, typename F>
constexpr size_t lanes_smem() {
    return (size_t)lanes_stages<WRITE_SCAN, F>() * lanes_tile<WRITE_SCAN, F>() * (4 + sizeof(F)) +
           (lanes_out<WRITE_SCAN, F>() ? lanes_tile<WRITE_SCAN, F>() * 4 : 0);
}
static_assert(lanes_smem<false, int32_t>() <= 227 * 1024 && lanes_smem<false, uint8_t>() <= 227 * 1024 &&
                  lanes_smem<true, int32_t>() <= 227 * 1024 && lanes_smem<true, uint8_t>() <= 227 * 1024,
              "shared memory");
// Segment sums staged per warp (the forms writing the scan with sums, where
// the shared memory left over allows at least 64 slots a warp, 2 KB kept for
// static shared memory): slots a warp, a multiple of 32, at most a warp's
// elements + 1. Measured (n = 2^26, Gelem/s, geometric / length-4 heads):
// scan + sums 406 / 334 -> 402 / 349, byte flags 544 / 386 -> 537 / 452;
// the byte-flag reduce gained nothing (639 / 476 -> 622 / 473) and does not
// stage.
#ifndef U32SCAN_S_STAGESUMS
#define U32SCAN_S_STAGESUMS 1
#endif
template <bool WRITE_SCAN, bool WANT_SUMS, typename F>
constexpr int lanes_sumcap() {
    constexpr long long spare = 227LL * 1024 - 2048 - (long long)lanes_smem<WRITE_SCAN, F>();
    constexpr long long cap = spare / (16 * 4) / 32 * 32;
    constexpr long long chunk = 128LL * lanes_r<WRITE_SCAN, F>() + 32;
    return (!U32SCAN_S_STAGESUMS || !WANT_SUMS || !WRITE_SCAN || cap < 64) ? 0 : (int)(cap < chunk ? cap : chunk);
}

// the smallest tile, which has the most tiles, sizes the workspace
constexpr unsigned long long min2(unsigned long long a, unsigned long long b) { return a < b ? a : b; }
constexpr unsigned long long kSTile = min2(min2(lanes_tile<false, int32_t>(), lanes_tile<false, uint8_t>()),
                                           min2(lanes_tile<true, int32_t>(), lanes_tile<true, uint8_t>()));

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
    constexpr unsigned long long TILE = lanes_tile<WRITE_SCAN, F>();
    const unsigned int n_tiles = (unsigned int)((n + head + TILE - 1) / TILE);
    constexpr int THREADS = 512;
    constexpr int SUMCAP = lanes_sumcap<WRITE_SCAN, WANT_SUMS, F>();
    auto kern = segscan_lanes_persistent<THREADS, lanes_r<WRITE_SCAN, F>(), lanes_stages<WRITE_SCAN, F>(), WRITE_SCAN,
                                         WANT_SUMS, F, lanes_out<WRITE_SCAN, F>(), SUMCAP>;
    constexpr size_t smem = lanes_smem<WRITE_SCAN, F>() + (size_t)16 * 4 * SUMCAP;
    static_assert(smem <= 227 * 1024 - 2048, "shared memory");
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
                                             aligned, skip_tile, limit_ns, tile_words_to_clear(ws_bytes));
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

extern "C" int u32scan_test_segscan_skip_publish(uint32_t *data, const int32_t *head_flags, size_t n,
                                                 uint32_t *seg_sums, size_t seg_capacity, uint32_t *nseg, void *ws,
                                                 size_t ws_bytes, unsigned int skip_tile, unsigned long long limit_ns,
                                                 u32scan_stream_t stream) {
    if (seg_sums != nullptr)
        return segscan_launch<true, true>(data, head_flags, n, seg_sums, seg_capacity, nseg, ws, ws_bytes,
                                          (cudaStream_t)stream, skip_tile, limit_ns);
    return segscan_launch<true, false>(data, head_flags, n, nullptr, 0, nseg, ws, ws_bytes, (cudaStream_t)stream,
                                       skip_tile, limit_ns);
}

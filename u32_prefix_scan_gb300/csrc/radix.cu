// radix.cu -- stable LSD radix-sort permutation of U32 keys.
//
// Source: the "parallel" package reference (entelechy docs), graph `sort`:
// the permutation that orders the keys, least significant bit first; per
// bit, sort_zeros counts the zeros at or before each place and sort_place
// sends a zero to its rank among the zeros and a one behind all the zeros at
// its rank among the ones ("the rank is the whole of what a stable radix
// pass needs"). The CAIRN "Concurrency" page, section "scan", builds its
// radix sort on an exclusive scan per digit the same way.
//
// Here a pass handles an 8-bit digit instead of one bit: a stable pass over
// a digit is the composition of the eight stable one-bit passes over its
// bits, so the result is the same unique stable permutation with 4 passes
// instead of 32. A histogram of all four digits, taken first in one read of
// the keys, gives every pass its digit bases (keys with a smaller digit
// value come first) and finds digits that are equal for every key, whose
// passes are skipped (exact: such a pass moves nothing); the histogram
// kernel's last block to finish derives both. Each digit pass is
// then one kernel over tiles of 11264 keys drawn in order: a tile ranks its
// keys stably within itself, publishes its 256 digit counts, and finds for
// every digit value the count of that value in all earlier tiles by a
// decoupled look-back (thread v walks back over the earlier tiles' words
// for value v, several a round trip, until one holds an inclusive count), so
// each key's slot is base + earlier count + rank; the tile is ordered by
// digit value in shared memory and written out run by run. Which passes run,
// and which buffers they read and write, is decided on the device, so the
// call stays asynchronous. The last pass writes the indices into `perm` and,
// for radix_sort_u32, the sorted keys into `keys_out`; a keys-only sort moves
// no indices at all. When only one digit varies, its pass orders one word a
// key (the key's place in the tile and its digit) and rebuilds the index and
// the key from it.
//
// Ranking. For the 32 keys of one warp round (one per lane), a per-warp
// table of lane masks, one word per value of the digit's low seven bits,
// and one ballot on its eighth bit give each lane the mask of lanes holding
// its digit value (each lane ORs its bit into its word of the table and
// reads the word back); the lowest lane of each value adds the value's
// count to the warp's running counter for it (one shared atomic add, whose
// old value is broadcast to the value's lanes) and clears the word, and a
// lane's rank is that old value plus the lanes below it in the mask. A round
// thus costs a few shared-memory accesses and little ALU work, which bounded
// the pass when the masks came from ballots. Each block asks L2 for the keys
// and indices of the tile drawn one resident grid later.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

// Digit-pass shape: threads per block, keys per thread per tile, resident
// blocks per SM (the launch bound); chosen by measurement on GB300 and
// overridable at build time for sweeps.
#ifndef U32SCAN_R_THREADS
#define U32SCAN_R_THREADS 512
#endif
#ifndef U32SCAN_R_KEYS
#define U32SCAN_R_KEYS 22
#endif
#ifndef U32SCAN_R_MINB
#define U32SCAN_R_MINB 2
#endif
constexpr int kRThreads = U32SCAN_R_THREADS;
constexpr int kRKeys = U32SCAN_R_KEYS;  // keys per thread per tile
constexpr unsigned int kRTile = kRThreads * kRKeys;
constexpr int kRWarps = kRThreads / 32;
constexpr unsigned int kRWarpKeys = 32 * kRKeys;  // a warp's run of the tile
static_assert(kRThreads >= 256 && kRThreads % 32 == 0 && kRKeys <= 32, "a thread per digit value; key bits fit a word");
static_assert(kRKeys >= 8, "the warps' match tables fit in the tile-ordered key buffer");
#ifndef U32SCAN_R_LOOK
#define U32SCAN_R_LOOK 4
#endif
constexpr int kRLook = U32SCAN_R_LOOK;  // earlier tiles read per look-back round trip
// 1: each block asks L2 for the tile one resident grid ahead.
#ifndef U32SCAN_R_PREFETCH
#define U32SCAN_R_PREFETCH 1
#endif
// Digit bits resolved by the match table (the rest by ballots): 2^TBITS
// words a warp; 7 measured 1 % faster than 8 (fewer bank conflicts on the
// table for one ballot), 4 to 6 slower.
#ifndef U32SCAN_R_TBITS
#define U32SCAN_R_TBITS 7
#endif
// One pass's role, decided on the device from the histograms.
struct RadixPlan {
    int active;  // this digit differs between keys
    int j;       // index of this pass among the active ones
    int m;       // number of active passes
    int pad;
};

// Workspace layout for n keys (all regions 256-byte aligned): the 256-byte
// header every operation keeps at offset 0 (tile counter, call epoch,
// device status), the histograms, the digit bases, the plan, one carry word
// per (tile, digit value), and the ping-pong buffers.
// Workspace of a sort of n keys. The histograms, digit bases, plan and
// ping-pong buffers hold small integers that could pass for another
// operation's tagged tile words, which lie in [header, reach). Far layout
// (the buffers at least as large as that span): the carry words first, then
// everything else from `reach` on, so the call leaves nothing but tagged
// words where other operations look and needs no clear at its end. Near
// layout (small sorts): everything packed after the header, and the call
// clears [header, reach) before it returns.
struct RadixLayout {
    size_t hist, done, bases, plan, desc, desc_end, k1, k2, i1, total, reach;
    unsigned int n_tiles;
    bool far;
    explicit RadixLayout(unsigned long long n) {
        n_tiles = (unsigned int)((n + kRTile - 1) / kRTile);
        reach = round_up(tile_word_reach(), 256);
        far = 12ull * n >= reach;
        const size_t desc_bytes = round_up(8ull * 256 * n_tiles, 256);
        size_t o = kHeaderBytes;
        if (far) {
            desc = o;
            o += desc_bytes;
            desc_end = o;
            o = o > reach ? o : reach;
        }
        hist = o;  // then the histogram kernel's count of finished blocks
        o += 4 * 256 * 4;
        done = o;
        o += 256;
        bases = o;
        o += round_up(4 * 256 * 4, 256);
        plan = o;
        o += round_up(4 * sizeof(RadixPlan), 256);
        if (!far) {
            desc = o;
            o += desc_bytes;
            desc_end = o;
        }
        k1 = o;
        o += round_up(4 * n, 256);
        k2 = o;
        o += round_up(4 * n, 256);
        i1 = o;
        o += round_up(4 * n, 256);
        total = o;
    }
};

// Counts of all four digits over all keys (one read), for the plan. One
// block of 1024 threads per SM. The counters are lane columns: row
// (digit, value) holds 32 words, one per lane, so the 32 atomic adds of a
// warp instruction always fall in 32 different banks whatever the keys.
constexpr int kHThreads = 1024;
constexpr size_t kHSmem = (size_t)4 * 256 * 32 * 4;  // 128 KiB

// The plan from the four complete histograms (called by every thread of
// one block; warp p < 4 takes digit p): a digit is constant when one value
// holds all n keys; each pass's base for digit value v is the number of
// keys whose digit is below v (an exclusive scan of that digit's
// histogram).
__device__ __forceinline__ void radix_plan_block(const unsigned int *hist, unsigned long long n, RadixPlan *plan,
                                                 unsigned int *bases) {
    __shared__ int s_active[4];
    const int lane = threadIdx.x & 31, p = threadIdx.x >> 5;
    if (p < 4) {
        // lane l holds digit values 8l .. 8l+7
        unsigned int c[8], sum = 0;
        bool whole = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = ld_relaxed_u32(hist + 256 * p + 8 * lane + i);
            sum += c[i];
            whole = whole || c[i] == n;
        }
        const bool active = !__any_sync(0xffffffffu, whole);
        unsigned int run = warp_inclusive_sum(sum, lane) - sum;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bases[256 * p + 8 * lane + i] = run;
            run += c[i];
        }
        if (lane == 0) s_active[p] = active ? 1 : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int j = 0, m = s_active[0] + s_active[1] + s_active[2] + s_active[3];
        for (int q = 0; q < 4; ++q) {
            plan[q].active = s_active[q];
            plan[q].j = j;
            plan[q].m = m;
            j += s_active[q];
        }
    }
}

// `done` counts the blocks that have added their counts (zero at launch);
// the last one computes the plan.
__global__ void __launch_bounds__(kHThreads, 1)
radix_histogram_kernel(const uint32_t *__restrict__ keys, unsigned long long n, unsigned int *hist,
                       unsigned int *done, RadixPlan *plan, unsigned int *bases) {
    extern __shared__ __align__(16) unsigned int h_cols[];  // [4 * 256][32]
    for (int i = threadIdx.x; i < 4 * 256 * 32; i += kHThreads) h_cols[i] = 0;
    __syncthreads();
    const unsigned int lane = threadIdx.x & 31;
    unsigned int *col = h_cols + lane;
    auto add = [&](uint32_t k) {
        atomicAdd(col + 32 * (k & 255u), 1u);
        atomicAdd(col + 32 * (256 + ((k >> 8) & 255u)), 1u);
        atomicAdd(col + 32 * (512 + ((k >> 16) & 255u)), 1u);
        atomicAdd(col + 32 * (768 + (k >> 24)), 1u);
    };
    auto add4 = [&](const uint4 &q) {
        add(q.x);
        add(q.y);
        add(q.z);
        add(q.w);
    };
    // scalar head up to 16-byte alignment, 16-byte body (four to eight loads
    // in flight a thread), scalar tail; n < 2^31 for a radix sort, so 32-bit
    // indices suffice
    const unsigned int n32 = (unsigned int)n;
    const unsigned int head = (unsigned int)((16 - (reinterpret_cast<uintptr_t>(keys) & 15)) & 15) / 4;
    const unsigned int h = head < n32 ? head : n32;
    const unsigned int nv = (n32 - h) / 4;
    const unsigned int gtid = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned int gstride = gridDim.x * blockDim.x;
    if (gtid < h) add(keys[gtid]);
    const uint4 *kv = reinterpret_cast<const uint4 *>(keys + h);
    unsigned int i = gtid;
    // software-pipelined: the next four loads are issued before the current
    // four are counted, so loads stay in flight through the atomics
    if (i + 3 * gstride < nv) {
        uint4 q0 = __ldcs(kv + i), q1 = __ldcs(kv + i + gstride), q2 = __ldcs(kv + i + 2 * gstride),
              q3 = __ldcs(kv + i + 3 * gstride);
        for (i += 4 * gstride; i + 3 * gstride < nv; i += 4 * gstride) {
            const uint4 n0 = __ldcs(kv + i), n1 = __ldcs(kv + i + gstride), n2 = __ldcs(kv + i + 2 * gstride),
                        n3 = __ldcs(kv + i + 3 * gstride);
            add4(q0);
            add4(q1);
            add4(q2);
            add4(q3);
            q0 = n0;
            q1 = n1;
            q2 = n2;
            q3 = n3;
        }
        add4(q0);
        add4(q1);
        add4(q2);
        add4(q3);
    }
    for (; i < nv; i += gstride) add4(__ldcs(kv + i));
    for (unsigned int j = h + 4 * nv + gtid; j < n32; j += gstride) add(keys[j]);
    __syncthreads();
    // thread r sums row r over the lanes, starting at its own lane's column
    // so that the 32 reads of a warp instruction fall in different banks
    for (int r = threadIdx.x; r < 4 * 256; r += kHThreads) {
        unsigned int sum = 0;
#pragma unroll 8
        for (int c = 0; c < 32; ++c) sum += h_cols[32 * r + ((c + (int)lane) & 31)];
        if (sum) atomicAdd(hist + r, sum);
    }
    __shared__ unsigned int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool last = atom_add_acq_rel(done, 1u) == gridDim.x - 1u;
        if (last) st_relaxed_u32(done, 0u);
        s_last = last ? 1u : 0u;
    }
    __syncthreads();
    if (s_last) radix_plan_block(hist, n, plan, bases);
}

// Buffers of one pass. Pass j of m active ones reads what pass j - 1 wrote
// (pass 0 reads the caller's keys and the identity permutation) and the
// last pass writes the results: indices into `perm` and, when sorted keys
// are wanted, keys into `keys_out`. Earlier passes alternate between a
// scratch buffer and the result buffer itself, counted back from the last
// pass so that it never reads the buffer it writes. Without keys_out the
// second key buffer is workspace (k2) and the last pass writes no keys;
// without perm no indices are moved at all.
struct PassBuffers {
    const uint32_t *in_keys;
    const int32_t *in_idx;  // null: the identity (first pass) or no indices
    uint32_t *out_keys;     // null: last pass of a permutation-only call
    int32_t *out_idx;       // null: keys-only sort
};

__device__ __forceinline__ PassBuffers pass_buffers(const RadixPlan &pl, const uint32_t *keys, uint32_t *k1,
                                                    uint32_t *k2, int32_t *i1, int32_t *perm,
                                                    uint32_t *keys_out) {
    PassBuffers b;
    const int j = pl.j, m = pl.m;
    uint32_t *klast = keys_out ? keys_out : k2;
    auto keys_of = [&](int q) -> uint32_t * {
        if (q == m - 1) return keys_out;  // null for a permutation-only call
        return ((m - 1 - q) & 1) ? k1 : klast;
    };
    auto idx_of = [&](int q) -> int32_t * {
        if (perm == nullptr) return nullptr;
        return q == m - 1 ? perm : (((m - 1 - q) & 1) ? i1 : perm);
    };
    b.in_keys = j == 0 ? keys : keys_of(j - 1);
    b.in_idx = j == 0 ? nullptr : idx_of(j - 1);
    b.out_keys = keys_of(j);
    b.out_idx = idx_of(j);
    return b;
}

// A thread's ranks (later tile positions), two 16-bit halves a word: both
// lie below the tile size. Halves are read and written by byte permutes.
constexpr int kRWords = (kRKeys + 1) / 2;
static_assert(kRTile <= 65536, "a tile position fits 16 bits");
__device__ __forceinline__ unsigned int rank_get(const unsigned int (&w)[kRWords], int r) {
    return (r & 1) ? (w[r >> 1] >> 16) : (w[r >> 1] & 0xffffu);
}
__device__ __forceinline__ void rank_set(unsigned int (&w)[kRWords], int r, unsigned int x) {
    w[r >> 1] = (r & 1) ? __byte_perm(w[r >> 1], x, 0x5410) : __byte_perm(w[r >> 1], x, 0x3254);
}

// Load this thread's keys of tile t (warp-striped: round r of warp w covers
// the 32 consecutive keys at t * kRTile + w * kRWarpKeys + 32 r) and rank
// them stably within the warp: afterwards rank r of wrank is the key's rank among
// the warp's keys of its digit value (in tile order) and s_wcnt[v] the
// warp's count of value v. FULL: every key of the tile lies in the array.
//
// A round finds the lanes holding each digit value through the warp's match
// table s_wmatch (2^U32SCAN_R_TBITS words, zero between rounds, indexed by
// the digit's low TBITS bits): every lane ORs its lane bit into its word and
// reads the word back, which, ANDed with ballots on the digit's other bits,
// is the mask of lanes sharing its value; the value's lowest lane then adds
// the count to the warp's counter and clears the word. (Eight ballots, one
// per digit bit, folded in every lane, measured slower: the fold costs
// about five ALU instructions a bit, and the pass was bound by the ALU
// pipe.)
template <bool FULL>
__device__ __forceinline__ unsigned int radix_rank_tile(const uint32_t *__restrict__ in_keys, unsigned int n32,
                                                        unsigned int wbase, int shift, uint32_t (&k)[kRKeys],
                                                        unsigned int (&wrank)[kRWords], unsigned int *s_wcnt,
                                                        unsigned int *s_wmatch, int lane) {
    unsigned int valid_bits = FULL ? 0xffffffffu : 0u;
#pragma unroll
    for (int r = 0; r < kRKeys; ++r) {
        const unsigned int e = wbase + 32u * r + (unsigned int)lane;
        if (FULL) {
            k[r] = __ldcs(in_keys + e);
        } else {
            k[r] = e < n32 ? __ldcs(in_keys + e) : 0u;
            valid_bits |= (e < n32 ? 1u : 0u) << r;
        }
    }
    for (int i = lane; i < 256; i += 32) {
        s_wcnt[i] = 0;
        s_wmatch[i] = 0;
    }
    __syncwarp();
    const unsigned int lanebit = 1u << lane;
#pragma unroll
    for (int r = 0; r < kRKeys; ++r) {
        const bool valid = FULL || ((valid_bits >> r) & 1u);
        const unsigned int d = (k[r] >> shift) & 255u;
        const unsigned int te = d & ((1u << U32SCAN_R_TBITS) - 1u);
        if (valid) atomicOr(s_wmatch + te, lanebit);
        unsigned int hi = 0xffffffffu;
#pragma unroll
        for (int b = U32SCAN_R_TBITS; b < 8; ++b) {
            const unsigned int bit = (d >> b) & 1u;
            hi &= __ballot_sync(0xffffffffu, bit != 0u) ^ (bit - 1u);
        }
        __syncwarp();  // every lane's bit is in before any lane reads
        const unsigned int same = valid ? (s_wmatch[te] & hi) : 0u;
        __syncwarp();  // every lane has read before a leader clears
        const unsigned int below = (unsigned int)__popc(same & lanemask_lt(lane));
        unsigned int old = 0;
        if (valid && below == 0) {
            old = atomicAdd(s_wcnt + d, (unsigned int)__popc(same));
            s_wmatch[te] = 0u;
        }
        const int leader = same ? __ffs(same) - 1 : 0;
        const unsigned int rk = __shfl_sync(0xffffffffu, old, leader) + below;
        if (r & 1)
            rank_set(wrank, r, rk);
        else
            wrank[r >> 1] = rk;  // the odd half is written next round
        __syncwarp();  // this round's counter updates and clears before the next round
    }
    return valid_bits;
}

// The 16-byte-aligned interior of [p, p + bytes), requested into L2.
__device__ __forceinline__ void prefetch_l2_interior(const void *p, unsigned long long bytes) {
    const uintptr_t a = (reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15);
    const uintptr_t e = (reinterpret_cast<uintptr_t>(p) + bytes) & ~uintptr_t(15);
    if (e > a) bulk_prefetch_l2(reinterpret_cast<const void *>(a), (unsigned int)(e - a));
}

// The identity permutation (and the keys unchanged) over this block's tile:
// the result when every digit is constant. Kept out of line so that the
// digit pass's own code is the same as without it.
__device__ __noinline__ void radix_identity_tile(const uint32_t *keys, int32_t *perm, uint32_t *keys_out,
                                                 unsigned long long n) {
    const unsigned long long lo = (unsigned long long)blockIdx.x * kRTile;
    const unsigned long long hi = lo + kRTile < n ? lo + kRTile : n;
    for (unsigned long long i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        if (perm) perm[i] = (int32_t)i;
        if (keys_out) keys_out[i] = keys[i];
    }
}

// One digit pass: tiles drawn in order; per tile: rank, carry each digit
// value's count across tiles by decoupled look-back, order the tile by digit
// value in shared memory, write each value's run of (key, index) pairs to
// consecutive slots. Carry word of (tile t, value v) at desc[256 t + v]
// (tile-major: the 32 values of a warp read 32 consecutive words for each
// earlier tile): the library's tagged format, value = the tile's count of v
// (aggregate) or the count of v in tiles 0..t (inclusive, P bit).
// One tile per block; `ahead`: tiles between a block's tile and the one it
// asks L2 for (the resident grid).
// One tile of a digit pass (the block's whole work). SINGLE: the only active
// pass (every other digit is equal for all keys): its indices are the
// identity, so a key is placed in shared memory as one word holding its
// place in the tile and its digit, and its index and key are rebuilt from
// that word when the tile is written (no second array of indices).
template <bool SINGLE>
__device__ __forceinline__ void radix_pass_tile(const PassBuffers &b, int p, unsigned long long n, unsigned int n_tiles,
                                                const unsigned int *__restrict__ bases, WsHeader *hdr,
                                                unsigned long long *desc, unsigned long long limit_ns,
                                                unsigned int ahead, unsigned long long clear_words) {
    // Shared memory (32-bit words): per-warp digit counters, later the warp
    // offsets in the tile-ordered buffer [kRWarps][256]; each value's run
    // start in the tile [256]; its first output slot minus that start [256];
    // the tile's keys in digit order [kRTile]; its indices in digit order
    // [kRTile].
    extern __shared__ __align__(128) unsigned int r_smem[];
    unsigned int(*s_cnt)[256] = reinterpret_cast<unsigned int(*)[256]>(r_smem);
    unsigned int *s_tileoff = r_smem + kRWarps * 256;
    unsigned int *s_delta = s_tileoff + 256;
    unsigned int *s_keys = s_delta + 256;
    int32_t *s_idx = reinterpret_cast<int32_t *>(s_keys + kRTile);
    __shared__ unsigned int s_part[kRWarps];
    __shared__ unsigned int s_t, s_epoch, s_kbase;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int shift = 8 * p;
    // n < 2^31 for a radix sort: 32-bit element indices
    const unsigned int n32 = (unsigned int)n;
    // Ask L2 for tile f's keys (and indices, when the pass moves them).
    auto prefetch_tile = [&](unsigned int f) {
        const unsigned int f0 = f * kRTile;
        const unsigned int cnt = n32 - f0 < kRTile ? n32 - f0 : kRTile;
        prefetch_l2_interior(b.in_keys + f0, 4ull * cnt);
        if (b.in_idx != nullptr && b.out_idx != nullptr) prefetch_l2_interior(b.in_idx + f0, 4ull * cnt);
    };
    if (threadIdx.x == 0) {
        unsigned int e;
        const unsigned int t = draw_tile(hdr, n_tiles, &e);
        s_t = t;
        s_epoch = e;
        if (U32SCAN_R_PREFETCH && ahead != 0u && t + ahead < n_tiles) prefetch_tile(t + ahead);
    }
    __syncthreads();
    const unsigned int t = s_t;
    const unsigned long long tag = tag_of(s_epoch);
    const unsigned int tile0 = t * kRTile;
    const bool full = n32 - tile0 >= kRTile;
    const unsigned int wbase = tile0 + (unsigned int)warp * kRWarpKeys;
    uint32_t k[kRKeys];
    unsigned int wrank[kRWords];
    // the warps' match tables live where the tile-ordered keys go later
    unsigned int *s_wmatch = s_keys + 256 * warp;
    const unsigned int valid_bits =
        full ? radix_rank_tile<true>(b.in_keys, n32, wbase, shift, k, wrank, s_cnt[warp], s_wmatch, lane)
             : radix_rank_tile<false>(b.in_keys, n32, wbase, shift, k, wrank, s_cnt[warp], s_wmatch, lane);
    __syncthreads();
    // Per digit value v (threads 0..255): warp offsets within the value's
    // run in this tile and the run's length, published at once.
    unsigned int tot = 0;
    unsigned long long *my = nullptr;
    if (threadIdx.x < 256) {
        const int v = threadIdx.x;
#pragma unroll
        for (int w = 0; w < kRWarps; ++w) {
            const unsigned int c = s_cnt[w][v];
            s_cnt[w][v] = tot;
            tot += c;
        }
        my = desc + 256ull * t + v;
        st_relaxed(my, tag | (t == 0 ? kFlagP : 0ull) | tot);
    }
    // The runs' starts in the tile: exclusive scan of the 256 run lengths.
    const unsigned int inc = warp_inclusive_sum(tot, lane);
    if (lane == 31 && threadIdx.x < 256) s_part[warp] = inc;
    __syncthreads();
    if (threadIdx.x < 256) {
        unsigned int pre = 0;
        for (int w = 0; w < warp; ++w) pre += s_part[w];
        const unsigned int start = pre + inc - tot;
        s_tileoff[threadIdx.x] = start;
        // each warp's first position for value v in the tile-ordered buffer
#pragma unroll
        for (int w = 0; w < kRWarps; ++w) s_cnt[w][threadIdx.x] += start;
    }
    __syncthreads();
    // Order the keys by digit value in shared memory; the ranks become each
    // key's position in the tile-ordered buffer. Then the indices: read from
    // the previous pass's buffer (all sixteen loads first, then the stores:
    // a load and its store taken in turn measured 16 % slower), or the
    // element indices on the first pass.
#pragma unroll
    for (int r = 0; r < kRKeys; ++r) {
        if (full || ((valid_bits >> r) & 1u)) {
            const unsigned int v = (k[r] >> shift) & 255u;
            const unsigned int pos = rank_get(wrank, r) + s_cnt[warp][v];
            if (SINGLE) {
                // the key's place in the tile (below 2^16) and its digit
                s_keys[pos] = ((unsigned int)warp * kRWarpKeys + 32u * r + (unsigned int)lane) | (v << 16);
            } else {
                rank_set(wrank, r, pos);
                s_keys[pos] = k[r];
            }
        }
    }
    // the digits every key shares (thread 0's first key is always in the array)
    if (SINGLE && threadIdx.x == 0) s_kbase = k[0] & ~(255u << shift);
    // The look-back's first window (threads 0..255, value v), loaded before
    // the indices are placed so that its round trip overlaps that work (4
    // words: 8 measured slower loaded here, and before the keys are placed
    // they spill).
    unsigned long long wd[kRLook];
    if (threadIdx.x < 256) {
        const unsigned long long *col = desc + threadIdx.x;
#pragma unroll
        for (int j = 0; j < kRLook; ++j) {
            const long long q = (long long)t - 1 - j;
            wd[j] = q >= 0 ? ld_relaxed(col + 256ull * (unsigned long long)q) : (tag | kFlagP);
        }
    }
    if (!SINGLE && b.out_idx) {
        int32_t idx[kRKeys];
#pragma unroll
        for (int r = 0; r < kRKeys; ++r) {
            const unsigned int e = wbase + 32u * r + (unsigned int)lane;
            idx[r] = b.in_idx ? ((full || ((valid_bits >> r) & 1u)) ? __ldcs(b.in_idx + e) : 0) : (int32_t)e;
        }
#pragma unroll
        for (int r = 0; r < kRKeys; ++r)
            if (full || ((valid_bits >> r) & 1u)) s_idx[rank_get(wrank, r)] = idx[r];
    }
    // Look back (threads 0..255, value v): the count of v in all earlier
    // tiles. Window word j holds tile pos - j (a virtual inclusive zero
    // before tile 0); fold from pos down to the first inclusive word; a word
    // not yet published ends the round, and the window is reloaded from it.
    if (threadIdx.x < 256) {
        const int v = threadIdx.x;
        const unsigned long long *col = desc + v;  // value v's word of tile q at col[256 q]
        unsigned int before = 0;
        long long pos = (long long)t - 1;
        unsigned long long t0 = 0;
        unsigned int iter = 0;
        while (true) {
            bool done = false, stalled = false;
            int used = 0;
#pragma unroll
            for (int j = 0; j < kRLook; ++j) {
                if (done || stalled) continue;
                if ((wd[j] & kTagMask) != tag) {
                    stalled = true;
                    continue;
                }
                before += (unsigned int)wd[j];
                ++used;
                if (wd[j] & kFlagP) done = true;
            }
            if (done) break;
            pos -= used;
            if (stalled) {  // a word not published yet: wait, bounded
                if (iter == 0) t0 = globaltimer();
                ++iter;
                if (iter >= 8) __nanosleep(64);
                if (iter >= kMaxSpinIters || globaltimer() - t0 > limit_ns) {
                    report_timeout(hdr, t);
                    break;
                }
            }
#pragma unroll
            for (int j = 0; j < kRLook; ++j)
                wd[j] = pos - j >= 0 ? ld_relaxed(col + 256ull * (unsigned long long)(pos - j)) : (tag | kFlagP);
        }
        if (t != 0) st_relaxed(my, tag | kFlagP | (before + tot));
        s_delta[v] = bases[256 * p + v] + before - s_tileoff[v];
    }
    __syncthreads();
    if (SINGLE) {
        // the index is the key's place (the identity before the only pass);
        // the key, the shared digits with its own
        const unsigned int count = full ? kRTile : n32 - tile0;
        const unsigned int kbase = s_kbase;
        for (unsigned int i = threadIdx.x; i < count; i += kRThreads) {
            const unsigned int w = s_keys[i];
            const unsigned int v = w >> 16;
            const unsigned int slot = s_delta[v] + i;
            if (b.out_keys) b.out_keys[slot] = kbase | (v << shift);
            if (b.out_idx) b.out_idx[slot] = (int32_t)(tile0 + (w & 0xffffu));
        }
    } else {
        const unsigned int count = full ? kRTile : n32 - tile0;
        for (unsigned int i = threadIdx.x; i < count; i += kRThreads) {
            const unsigned int key = s_keys[i];
            const unsigned int slot = s_delta[(key >> shift) & 255u] + i;
            if (b.out_keys) b.out_keys[slot] = key;
            if (b.out_idx) b.out_idx[slot] = s_idx[i];
        }
    }
    // A launch that ends a tag period zeroes the first clear_words tile
    // words (far layout: every word another operation may read; the sort's
    // own buffers lie past them). Near layout: 0, the call clears at its end.
    finish_period(hdr, s_epoch, reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(hdr) + kHeaderBytes),
                  clear_words);
}

// The single-pass tile. (Kept out of line, the call cost the other passes'
// code a spill and 5 % of their time.)
__device__ __forceinline__ void radix_pass_tile_single(int p, const uint32_t *keys, int32_t *perm, uint32_t *keys_out,
                                                    unsigned long long n, unsigned int n_tiles,
                                                    const unsigned int *__restrict__ bases, WsHeader *hdr,
                                                    unsigned long long *desc, unsigned long long limit_ns,
                                                    unsigned int ahead, unsigned long long clear_words) {
    // the only pass reads the caller's keys and writes the results
    const PassBuffers b{keys, nullptr, keys_out, perm};
    radix_pass_tile<true>(b, p, n, n_tiles, bases, hdr, desc, limit_ns, ahead, clear_words);
}

__global__ void __launch_bounds__(kRThreads, U32SCAN_R_MINB)
radix_onesweep_kernel(const RadixPlan *__restrict__ plan, int p, const uint32_t *keys, uint32_t *k1, uint32_t *k2,
                      int32_t *i1, int32_t *perm, uint32_t *keys_out, unsigned long long n, unsigned int n_tiles,
                      const unsigned int *__restrict__ bases, WsHeader *hdr, unsigned long long *desc,
                      unsigned long long limit_ns, unsigned int ahead, unsigned long long clear_words) {
    const RadixPlan pl = plan[p];
    if (!pl.active) {
        // Every digit constant (every key equal): the permutation is the
        // identity, written by the last digit's launch.
        if (p == 3 && pl.m == 0) radix_identity_tile(keys, perm, keys_out, n);
        return;
    }
    if (pl.m == 1) {
        radix_pass_tile_single(p, keys, perm, keys_out, n, n_tiles, bases, hdr, desc, limit_ns, ahead, clear_words);
    } else {
        const PassBuffers b = pass_buffers(pl, keys, k1, k2, i1, perm, keys_out);
        radix_pass_tile<false>(b, p, n, n_tiles, bases, hdr, desc, limit_ns, ahead, clear_words);
    }
}

constexpr size_t kRSmem = (size_t)(kRWarps * 256 + 512 + 2 * kRTile) * 4;

size_t radix_workspace_bytes(unsigned long long n) { return RadixLayout(n).total; }

static int radix_launch(const uint32_t *keys, unsigned long long n, int32_t *perm, uint32_t *keys_out, void *ws,
                        size_t ws_bytes, cudaStream_t stream) {
    if (n >= (1ull << 31)) return U32SCAN_EINVAL;
    if (n > 0 && (keys == nullptr || (perm == nullptr && keys_out == nullptr))) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(keys) & 3) || (reinterpret_cast<uintptr_t>(perm) & 3) ||
        (reinterpret_cast<uintptr_t>(keys_out) & 3))
        return U32SCAN_EINVAL;
    if (keys_out != nullptr && n > 0 &&
        reinterpret_cast<const char *>(keys_out) < reinterpret_cast<const char *>(keys + n) &&
        reinterpret_cast<const char *>(keys) < reinterpret_cast<const char *>(keys_out + n))
        return U32SCAN_EINVAL;  // the sorted keys may not overlap the input
    if (n == 0) return U32SCAN_OK;
    const RadixLayout L(n);
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < L.total) return U32SCAN_EWORKSPACE;
    char *w = static_cast<char *>(ws);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(w);
    unsigned int *hist = reinterpret_cast<unsigned int *>(w + L.hist);
    unsigned int *done = reinterpret_cast<unsigned int *>(w + L.done);
    unsigned int *bases = reinterpret_cast<unsigned int *>(w + L.bases);
    RadixPlan *plan = reinterpret_cast<RadixPlan *>(w + L.plan);
    unsigned long long *desc = reinterpret_cast<unsigned long long *>(w + L.desc);
    uint32_t *k1 = reinterpret_cast<uint32_t *>(w + L.k1);
    uint32_t *k2 = reinterpret_cast<uint32_t *>(w + L.k2);
    int32_t *i1 = reinterpret_cast<int32_t *>(w + L.i1);
    // per device, once: shared-memory limits, SM count, resident digit-pass blocks
    int sms = 0, resident = 0;
    {
        static std::mutex mu;
        static int dev_sms[64], dev_resident[64];
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
        std::lock_guard<std::mutex> lock(mu);
        if (dev_sms[dev] == 0) {
            int s = 0, bps = 0;
            if (cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaFuncSetAttribute(radix_onesweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kRSmem) != cudaSuccess ||
                cudaFuncSetAttribute(radix_histogram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kHSmem) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, radix_onesweep_kernel, kRThreads, kRSmem) !=
                    cudaSuccess)
                return U32SCAN_ECUDA;
            dev_resident[dev] = s * (bps > 0 ? bps : 1);
            dev_sms[dev] = s;
        }
        sms = dev_sms[dev];
        resident = dev_resident[dev];
    }
    // the histograms and the finished-block count (one memset: they are adjacent)
    if (cudaMemsetAsync(hist, 0, L.bases - L.hist, stream) != cudaSuccess) return U32SCAN_ECUDA;
    // The digit passes' carry words (each pass's launch has its own tag).
    // Where other operations keep tile words, the words can only be tagged
    // or zero; past that span another call's histograms or buffers may lie.
    {
        const size_t from = L.far ? (L.desc > L.reach ? L.desc : L.reach) : L.desc;
        if (L.desc_end > from)
            if (const int rc = clear_tile_words(w + from, L.desc_end - from, stream); rc != U32SCAN_OK) return rc;
    }
    radix_histogram_kernel<<<sms, kHThreads, kHSmem, stream>>>(keys, n, hist, done, plan, bases);
    const unsigned long long clear_words = L.far ? tile_words_to_clear(ws_bytes) : 0ull;
    for (int p = 0; p < 4; ++p)
        radix_onesweep_kernel<<<L.n_tiles, kRThreads, kRSmem, stream>>>(plan, p, keys, k1, k2, i1, perm, keys_out, n,
                                                                         L.n_tiles, bases, hdr, desc, kDefaultLimitNs,
                                                                         (unsigned int)resident, clear_words);
    if (cudaGetLastError() != cudaSuccess) return U32SCAN_ECUDA;
    if (L.far) return U32SCAN_OK;
    // Near layout: leave no data where another operation's tile words may
    // go (the histograms, bases and ping-pong buffers lie there). The whole
    // of that span is zeroed, not only this call's part of it, which also
    // serves as the end of a tag period if one of the passes ended one.
    const size_t end = ws_bytes < L.reach ? ws_bytes : L.reach;
    return clear_tile_words(w + kHeaderBytes, end - kHeaderBytes, stream);
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int radix_sort_perm_u32(const uint32_t *keys, size_t n, int32_t *perm, void *ws, size_t ws_bytes,
                                   u32scan_stream_t stream) {
    if (n > 0 && perm == nullptr) return U32SCAN_EINVAL;
    return radix_launch(keys, n, perm, nullptr, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int radix_sort_u32(const uint32_t *keys, size_t n, uint32_t *keys_out, int32_t *perm, void *ws,
                              size_t ws_bytes, u32scan_stream_t stream) {
    if (n > 0 && keys_out == nullptr) return U32SCAN_EINVAL;
    return radix_launch(keys, n, perm, keys_out, ws, ws_bytes, (cudaStream_t)stream);
}

// scan.cu -- device-wide U32 prefix sum, exclusive and inclusive, in place.
//
// Source: "scan.bend source" (bendlib), section API: `exclusive` makes a[j]
// the sum a[0] + .. + a[j-1] and `inclusive` the sum through a[j]; both
// return the total, and sums wrap at 2^32 (header comment). The page's
// three passes (block sums, scan of the sums, rescan from each base) read
// the data twice; here one kernel reads each element once and writes it
// once, carrying tile prefixes with the single-pass look-back of
// internal.cuh.
//
// Tile layout. A tile is THREADS * V * 4 consecutive elements. Warp w owns
// the w-th run of 128 * V elements; its lane l holds, for r = 0 .. V-1, the
// four elements starting at 128 * r + 4 * l of that run. Each of the V
// 16-byte loads of a warp therefore covers 512 contiguous bytes. Scan order
// inside the warp is r-major: a warp-wide scan of the per-lane sums for
// r = 0, then r = 1 carried on, and so on.
//
// Alignment. Elements are addressed by a virtual index v = i + head, where
// head = (address of a[0] mod 16) / 4, so that virtual multiples of 4 are
// 16-byte aligned. Tiles cover virtual ranges; a tile wholly inside
// [head, head + n) uses 16-byte loads and stores, the (at most two) others
// use guarded scalar accesses.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

// Persistent launch shape (threads, u32x4 loads per thread per tile, ring
// stages, look-back words per lane, minimum resident blocks per SM); the
// defaults were chosen by measurement on GB300 and can be overridden at
// build time for tuning sweeps.
#ifndef U32SCAN_P_THREADS
#define U32SCAN_P_THREADS 512
#endif
#ifndef U32SCAN_P_V
#define U32SCAN_P_V 8
#endif
#ifndef U32SCAN_P_STAGES
#define U32SCAN_P_STAGES 2
#endif
#ifndef U32SCAN_P_LOOK
#define U32SCAN_P_LOOK 1
#endif
// 1: a full tile's results are written to a shared-memory buffer and stored
// by one 1-D bulk copy (TMA); 0: 16-byte streaming stores from registers.
#ifndef U32SCAN_P_BULKSTORE
#define U32SCAN_P_BULKSTORE 1
#endif
#ifndef U32SCAN_P_MINB
#define U32SCAN_P_MINB 1
#endif

namespace u32scan {

// Per-round warp scan of a tile held in registers (layout above), under OP:
// x becomes the scan relative to the warp's start; returns the warp's fold.
template <int V, bool INCLUSIVE, int OP>
__device__ __forceinline__ unsigned int warp_scan_rounds(uint4 (&x)[V], int lane) {
    using M = Monoid<OP>;
    unsigned int carry = M::identity();
#pragma unroll
    for (int r = 0; r < V; ++r) {
        const unsigned int sum = M::apply(M::apply(x[r].x, x[r].y), M::apply(x[r].z, x[r].w));
        const unsigned int inc = M::warp_inclusive(sum, lane);
        const unsigned int ex = M::apply(carry, M::warp_exclusive(inc, sum, lane));
        if (INCLUSIVE) {
            x[r].x = M::apply(ex, x[r].x);
            x[r].y = M::apply(x[r].x, x[r].y);
            x[r].z = M::apply(x[r].y, x[r].z);
            x[r].w = M::apply(x[r].z, x[r].w);
        } else {
            const unsigned int a = x[r].x, b = x[r].y, c = x[r].z;
            x[r].x = ex;
            x[r].y = M::apply(ex, a);
            x[r].z = M::apply(x[r].y, b);
            x[r].w = M::apply(x[r].z, c);
        }
        carry = M::apply(carry, __shfl_sync(0xffffffffu, inc, 31));
    }
    return carry;
}

// One tile per block, for short arrays: enough blocks to fill the GPU.
template <int THREADS, int V, bool INCLUSIVE, int OP>
__global__ void __launch_bounds__(THREADS, (THREADS >= 512 ? 2 : 4))
scan_u32_kernel(uint32_t *__restrict__ data, unsigned long long n, uint32_t *total, const uint32_t *carry_in,
                WsHeader *hdr,
                unsigned long long *desc, unsigned int n_tiles, unsigned int head, unsigned int skip_tile,
                unsigned long long limit_ns, unsigned long long clear_words) {
    using M = Monoid<OP>;
    constexpr int WARPS = THREADS / 32;
    constexpr unsigned long long TILE = (unsigned long long)THREADS * V * 4;
    static_assert(WARPS <= 32, "one warp scans the warp totals");
    __shared__ unsigned int s_tile, s_epoch;
    __shared__ unsigned int s_warp[WARPS];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        unsigned int e;
        s_tile = draw_tile(hdr, n_tiles, &e);
        s_epoch = e;
    }
    __syncthreads();
    const unsigned int t = s_tile;
    const unsigned long long tag = tag_of(s_epoch);

    // Tile-local element index of this lane's first element, and the
    // tile-local range [lo, hi) that lies inside the array.
    const unsigned long long tile_v0 = (unsigned long long)t * TILE;
    const unsigned int li0 = (unsigned int)warp * (128 * V) + 4u * (unsigned int)lane;
    const unsigned int lo = tile_v0 < head ? (unsigned int)(head - tile_v0) : 0u;
    const unsigned long long left = head + n - tile_v0;
    const unsigned int hi = left < TILE ? (unsigned int)left : (unsigned int)TILE;
    const bool full = lo == 0 && hi == TILE;
    // Address of the tile's virtual element 0 (16-byte aligned); element
    // li of the tile is tbase[li]. Only in-range elements are dereferenced.
    uint32_t *tbase = reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(data) - 4ull * head) + tile_v0;

    uint4 x[V];
    if (full) {
#pragma unroll
        for (int r = 0; r < V; ++r) x[r] = __ldcs(reinterpret_cast<const uint4 *>(tbase + li0 + 128 * r));
    } else {
#pragma unroll
        for (int r = 0; r < V; ++r) {
            unsigned int e[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const unsigned int li = li0 + 128 * r + c;
                e[c] = (li >= lo && li < hi) ? tbase[li] : M::identity();
            }
            x[r] = make_uint4(e[0], e[1], e[2], e[3]);
        }
    }
    const unsigned int wtot = warp_scan_rounds<V, INCLUSIVE, OP>(x, lane);
    if (lane == 0) s_warp[warp] = wtot;
    __syncthreads();

    if (warp == 0) {
        const unsigned int wt = lane < WARPS ? s_warp[lane] : M::identity();
        const unsigned int winc = M::warp_inclusive(wt, lane);
        const unsigned int agg = __shfl_sync(0xffffffffu, winc, 31);
        const unsigned int wex = M::warp_exclusive(winc, wt, lane);
        const bool publish = t != skip_tile;
        // Everything before the array folds into tile 0: the carry-in, else the identity.
        const unsigned int cin = (t == 0 && carry_in != nullptr) ? *carry_in : M::identity();
        if (lane == 0 && publish) publish_aggregate(desc, t, M::apply(cin, agg), tag);
        unsigned long long win[1];
        lookback_window<1, OP>(desc, (long long)t - 1, tag, lane, win);
        const unsigned int prefix =
            M::apply(cin, lookback_prefix_wide<1, OP>(desc, t, tag, hdr, limit_ns, lane, win));
        if (lane == 0 && publish && t != 0) publish_inclusive(desc, t, M::apply(prefix, agg), tag);
        if (lane < WARPS) s_warp[lane] = M::apply(prefix, wex);
        if (t == n_tiles - 1u && lane == 0 && total != nullptr) *total = M::apply(prefix, agg);
    }
    __syncthreads();

    const unsigned int base = s_warp[warp];
#pragma unroll
    for (int r = 0; r < V; ++r) {
        x[r].x = M::apply(base, x[r].x);
        x[r].y = M::apply(base, x[r].y);
        x[r].z = M::apply(base, x[r].z);
        x[r].w = M::apply(base, x[r].w);
    }
    if (full) {
#pragma unroll
        for (int r = 0; r < V; ++r) __stcs(reinterpret_cast<uint4 *>(tbase + li0 + 128 * r), x[r]);
    } else {
#pragma unroll
        for (int r = 0; r < V; ++r) {
            const unsigned int e[4] = {x[r].x, x[r].y, x[r].z, x[r].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const unsigned int li = li0 + 128 * r + c;
                if (li >= lo && li < hi) tbase[li] = e[c];
            }
        }
    }
    finish_period(hdr, s_epoch, desc, clear_words);
}

// Persistent form for long arrays. Each block loops over tiles drawn from
// the tile counter, keeping S tiles in flight: tile loads are 1-D bulk
// copies (TMA) into an S-deep ring of shared-memory stages, each completing
// on its own mbarrier, so global loads keep streaming while the block waits
// on a predecessor's carry.
//
// The block is software-pipelined by one tile: in each round it scans the
// next tile locally and publishes that tile's aggregate, then walks the
// look-back of the current tile (whose aggregate went out a round earlier),
// adds the prefix and stores it. Aggregates thus appear one round before any
// tile needs them, and a look-back never waits on a neighbour that is
// merely behind in its own queue.
//
// Tiles are drawn in globally increasing order and each block processes its
// draws in order, so every predecessor of a waiting tile is held by a running
// block that publishes it (forward progress). Each block draws exactly S
// indices past the last tile; the draw of n_tiles + S * gridDim.x - 1 is the
// last of the launch and re-arms the header.
template <int THREADS, int V, int S, int K, bool INCLUSIVE, int OP>
__global__ void __launch_bounds__(THREADS, U32SCAN_P_MINB)
scan_u32_persistent(uint32_t *__restrict__ data, unsigned long long n, uint32_t *total, const uint32_t *carry_in,
                    WsHeader *hdr,
                    unsigned long long *desc, unsigned int n_tiles, unsigned int head, unsigned int skip_tile,
                    unsigned long long limit_ns, unsigned long long clear_words) {
    using M = Monoid<OP>;
    constexpr int WARPS = THREADS / 32;
    constexpr unsigned int TILE = THREADS * V * 4;
    constexpr unsigned int TILE_BYTES = TILE * 4;
    static_assert(WARPS <= 32, "one warp scans the warp totals");
    static_assert(S >= 2, "the pipeline reads one stage ahead");
    extern __shared__ __align__(128) uint4 stage_buf[];  // S stages of TILE elements (+ the output buffer)
    __shared__ __align__(8) unsigned long long bar[S];
    __shared__ unsigned int s_tile[S];
    __shared__ unsigned int s_wt[2][WARPS];  // warp totals of the current / next tile
    __shared__ unsigned int s_base[WARPS];   // per-warp prefix of the current tile
    __shared__ unsigned int s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned int last_draw = n_tiles + (unsigned int)S * gridDim.x - 1u;
    uint32_t *vbase = reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(data) - 4ull * head);
    // The producer (lane 0 of the last warp) draws tiles and starts their
    // copies, so its atomic round trip stays off warp 0's look-back path.
    const bool producer = threadIdx.x == THREADS - 32;
    unsigned int latest_parity = 0;  // producer: bit st = phase parity of stage st's latest draw

    auto tile_full = [&](unsigned int id) {
        const unsigned long long v0 = (unsigned long long)id * TILE;
        return v0 >= head && v0 + TILE <= head + n;
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
            mbar_arrive_expect_tx(b, TILE_BYTES);
            bulk_load(smem_u32(stage_buf + st * (TILE / 4)), vbase + (unsigned long long)id * TILE, TILE_BYTES, b);
        } else {
            mbar_arrive(b);  // nothing to copy: a partial tile reads global memory, a past-the-end draw stops
        }
    };
    const unsigned int li0 = (unsigned int)warp * (128 * V) + 4u * (unsigned int)lane;
    volatile unsigned int *vs_tile = s_tile;
    // The fold of everything before tile t's array start: the carry-in for
    // tile 0 (when given), the identity otherwise.
    auto carry_of = [&](unsigned int t) -> unsigned int {
        return (t == 0 && carry_in != nullptr) ? *carry_in : M::identity();
    };

    // Read draw number u (stage u % S) into x and scan it per warp; the warp
    // totals go to s_wt[u & 1]. Returns the tile index, n_tiles if the draw
    // is past the end, or n_tiles + 1 if its copy timed out.
    auto read_tile = [&](unsigned int u, uint4 (&x)[V]) -> unsigned int {
        const int st = (int)(u % S);
        if (!mbar_wait_bounded(smem_u32(&bar[st]), (u / S) & 1u, limit_ns)) {
            report_timeout(hdr, 0xfffffffeu);
            return n_tiles + 1u;
        }
        const unsigned int t = vs_tile[st];
        if (t >= n_tiles) return n_tiles;
        const unsigned long long tile_v0 = (unsigned long long)t * TILE;
        if (tile_full(t)) {
            const uint4 *sb = stage_buf + st * (TILE / 4) + (li0 >> 2);
#pragma unroll
            for (int r = 0; r < V; ++r) x[r] = sb[32 * r];
        } else {
            const unsigned int lo = tile_v0 < head ? (unsigned int)(head - tile_v0) : 0u;
            const unsigned long long left = head + n - tile_v0;
            const unsigned int hi = left < TILE ? (unsigned int)left : TILE;
            const uint32_t *tb = vbase + tile_v0;
#pragma unroll
            for (int r = 0; r < V; ++r) {
                unsigned int e[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const unsigned int li = li0 + 128 * r + c;
                    e[c] = (li >= lo && li < hi) ? tb[li] : M::identity();
                }
                x[r] = make_uint4(e[0], e[1], e[2], e[3]);
            }
        }
        const unsigned int wtot = warp_scan_rounds<V, INCLUSIVE, OP>(x, lane);
        if (lane == 0) s_wt[u & 1][warp] = wtot;
        return t;
    };
    // Store the current tile. With bulk stores, a full tile goes through the
    // output buffer after the S stages: every thread writes its part, a
    // barrier, then thread 0 starts one 1-D bulk copy of the whole tile (its
    // previous copy has finished reading the buffer: thread 0 waited for
    // that before barrier B). tile_full(t) is the same for every thread.
    auto store_tile = [&](unsigned int t, const uint4 (&x)[V], unsigned int base) {
        const unsigned long long tile_v0 = (unsigned long long)t * TILE;
        uint32_t *tb = vbase + tile_v0;
        if (tile_full(t)) {
            if (U32SCAN_P_BULKSTORE) {
                uint4 *ob = stage_buf + S * (TILE / 4);
#pragma unroll
                for (int r = 0; r < V; ++r)
                    ob[(li0 >> 2) + 32 * r] = make_uint4(M::apply(base, x[r].x), M::apply(base, x[r].y), M::apply(base, x[r].z), M::apply(base, x[r].w));
                fence_proxy_async_smem();
                __syncthreads();  // barrier C: the output buffer is complete
                if (threadIdx.x == 0) bulk_store(tb, smem_u32(ob), TILE_BYTES);
            } else {
#pragma unroll
                for (int r = 0; r < V; ++r) {
                    const uint4 y = make_uint4(M::apply(base, x[r].x), M::apply(base, x[r].y), M::apply(base, x[r].z), M::apply(base, x[r].w));
                    __stcs(reinterpret_cast<uint4 *>(tb + li0 + 128 * r), y);
                }
            }
        } else {
            const unsigned int lo = tile_v0 < head ? (unsigned int)(head - tile_v0) : 0u;
            const unsigned long long left = head + n - tile_v0;
            const unsigned int hi = left < TILE ? (unsigned int)left : TILE;
#pragma unroll
            for (int r = 0; r < V; ++r) {
                const unsigned int e[4] = {x[r].x, x[r].y, x[r].z, x[r].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const unsigned int li = li0 + 128 * r + c;
                    if (li >= lo && li < hi) tb[li] = M::apply(base, e[c]);
                }
            }
        }
    };
    // Warp 0: block aggregate of the tile whose warp totals are in s_wt[slot];
    // returns it, and leaves in wex this lane's exclusive warp offset.
    auto block_aggregate = [&](int slot, unsigned int &wex) -> unsigned int {
        const unsigned int wt = lane < WARPS ? s_wt[slot][lane] : M::identity();
        const unsigned int winc = M::warp_inclusive(wt, lane);
        wex = M::warp_exclusive(winc, wt, lane);
        return __shfl_sync(0xffffffffu, winc, 31);
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

    // Prologue: read draw 0.
    uint4 xc[V], xn[V];
    unsigned int tc = read_tile(0, xc);
    unsigned int agg_c = 0, wex_c = 0;
    if (!__syncthreads_or(tc >= n_tiles)) {
        if (producer) {
            fence_proxy_async_smem();
            issue(0);
            latest_parity ^= 1u;
        }
        if (warp == 0) {
            agg_c = block_aggregate(0, wex_c);
            if (lane == 0 && tc != skip_tile) publish_aggregate(desc, tc, M::apply(carry_of(tc), agg_c), tag);
        }
        for (unsigned int u = 1;; ++u) {
            // Look ahead: read draw u and publish its aggregate.
            const unsigned int tn = read_tile(u, xn);
            const bool more = !__syncthreads_or(tn >= n_tiles);  // barrier A
            unsigned int agg_n = 0, wex_n = 0;
            if (more && producer) {
                fence_proxy_async_smem();
                const int st = (int)(u % S);
                issue(st);
                latest_parity ^= 1u << st;
            }
            if (warp == 0) {
                if (more) {
                    agg_n = block_aggregate((int)(u & 1), wex_n);
                    if (lane == 0 && tn != skip_tile) publish_aggregate(desc, tn, M::apply(carry_of(tn), agg_n), tag);
                }
                // Finish the current tile: its look-back, inclusive prefix, bases.
                unsigned long long win[K];
                lookback_window<K, OP>(desc, (long long)tc - 1, tag, lane, win);
                const unsigned int prefix =
                    M::apply(carry_of(tc), lookback_prefix_wide<K, OP>(desc, tc, tag, hdr, limit_ns, lane, win));
                if (lane == 0 && tc != 0 && tc != skip_tile)
                    publish_inclusive(desc, tc, M::apply(prefix, agg_c), tag);
                if (lane < WARPS) s_base[lane] = M::apply(prefix, wex_c);
                if (tc == n_tiles - 1u && lane == 0 && total != nullptr) *total = M::apply(prefix, agg_c);
            }
            if (U32SCAN_P_BULKSTORE && threadIdx.x == 0) bulk_wait_read();  // output buffer free again
            __syncthreads();  // barrier B: bases of the current tile are visible
            store_tile(tc, xc, s_base[warp]);
            if (!more) break;
#pragma unroll
            for (int r = 0; r < V; ++r) xc[r] = xn[r];
            tc = tn;
            agg_c = agg_n;
            wex_c = wex_n;
        }
    }
    // Leave no bulk copy in flight into or out of this block's shared
    // memory: wait (bounded) for the latest phase of every stage (on the
    // normal path the outstanding draws are past the end and completed
    // already), and for thread 0's bulk stores.
    if (producer) {
#pragma unroll
        for (int st = 0; st < S; ++st)
            (void)mbar_wait_bounded(smem_u32(&bar[st]), (latest_parity >> st) & 1u, limit_ns);
    }
    if (U32SCAN_P_BULKSTORE && threadIdx.x == 0) bulk_wait_all();
    finish_period(hdr, s_epoch, desc, clear_words);
}

// Launch shapes, chosen by n: long arrays use the persistent kernel, short
// ones the one-tile-per-block kernel (narrow tiles, enough blocks).
constexpr int kPThreads = U32SCAN_P_THREADS, kPV = U32SCAN_P_V, kPStages = U32SCAN_P_STAGES,
              kPLook = U32SCAN_P_LOOK;
constexpr unsigned long long kPTile = (unsigned long long)kPThreads * kPV * 4;
constexpr size_t kPSmem = (size_t)(kPStages + (U32SCAN_P_BULKSTORE ? 1 : 0)) * kPTile * 4;
#ifndef U32SCAN_P_MINN_LOG2
#define U32SCAN_P_MINN_LOG2 19  // arrays of at least 2^this elements take the persistent kernel
#endif
constexpr unsigned long long kPersistentMinN = 1ull << U32SCAN_P_MINN_LOG2;

struct ScanShape {
    bool persistent;
    int threads, v;
    unsigned long long tile() const { return (unsigned long long)threads * v * 4; }
};

static ScanShape scan_shape(unsigned long long n) {
    if (n >= kPersistentMinN) return {true, kPThreads, kPV};
    return {false, 256, 2};
}

size_t scan_workspace_bytes(unsigned long long n) {
    const unsigned long long tiles = (n + 3 + scan_shape(n).tile() - 1) / scan_shape(n).tile();
    return round_up(kHeaderBytes + 8 * tiles, 256);
}

static const unsigned int kOne = 1u;  // the multiply identity, copied to `total` when n == 0

// Per-device launch facts for the persistent kernels, looked up once.
struct DeviceFacts {
    int sms = 0;
    int blocks_per_sm[2][7] = {};
};
static std::mutex g_facts_mu;
static DeviceFacts g_facts[64];

template <bool INCLUSIVE, int OP>
static int persistent_grid(int *grid_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    std::lock_guard<std::mutex> lock(g_facts_mu);
    DeviceFacts &f = g_facts[dev];
    if (f.sms == 0 && cudaDeviceGetAttribute(&f.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return U32SCAN_ECUDA;
    int &bps = f.blocks_per_sm[INCLUSIVE ? 1 : 0][OP];
    if (bps == 0) {
        auto kern = scan_u32_persistent<kPThreads, kPV, kPStages, kPLook, INCLUSIVE, OP>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmem) != cudaSuccess)
            return U32SCAN_ECUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, kPThreads, kPSmem) != cudaSuccess || bps < 1)
            return U32SCAN_ECUDA;
    }
    *grid_out = f.sms * bps;
    return U32SCAN_OK;
}

template <bool INCLUSIVE, int OP = kAdd>
static int scan_launch(uint32_t *data, unsigned long long n, uint32_t *total, void *ws, size_t ws_bytes,
                       cudaStream_t stream, unsigned int skip_tile, unsigned long long limit_ns,
                       const uint32_t *carry_in = nullptr) {
    if ((n > 0 && data == nullptr) || n >= (1ull << 32)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(data) & 3) || (reinterpret_cast<uintptr_t>(total) & 3))
        return U32SCAN_EINVAL;
    if (n == 0) {
        if (total && carry_in) {  // nothing after the carry-in: the fold is the carry-in
            if (cudaMemcpyAsync(total, carry_in, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
                return U32SCAN_ECUDA;
        } else if (total) {  // the fold of nothing is the operator's identity
            const unsigned int id = OP == kMul ? 1u : (OP == kAnd || OP == kMin) ? 0xffffffffu : 0u;
            if (cudaMemsetAsync(total, id ? 0xff : 0, sizeof(uint32_t), stream) != cudaSuccess) return U32SCAN_ECUDA;
            if (id == 1u && cudaMemcpyAsync(total, &kOne, sizeof(uint32_t), cudaMemcpyHostToDevice, stream) != cudaSuccess)
                return U32SCAN_ECUDA;
        }
        return U32SCAN_OK;
    }
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < scan_workspace_bytes(n))
        return U32SCAN_EWORKSPACE;
    const ScanShape sh = scan_shape(n);
    const unsigned int head = (unsigned int)((reinterpret_cast<uintptr_t>(data) & 15) >> 2);
    const unsigned int n_tiles = (unsigned int)((n + head + sh.tile() - 1) / sh.tile());
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    unsigned long long *desc = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kHeaderBytes);
    const unsigned long long clear_words = tile_words_to_clear(ws_bytes);
    if (sh.persistent) {
        int grid = 0;
        const int rc = persistent_grid<INCLUSIVE, OP>(&grid);
        if (rc != U32SCAN_OK) return rc;
        if ((unsigned int)grid > n_tiles) grid = (int)n_tiles;
        scan_u32_persistent<kPThreads, kPV, kPStages, kPLook, INCLUSIVE, OP><<<grid, kPThreads, kPSmem, stream>>>(
            data, n, total, carry_in, hdr, desc, n_tiles, head, skip_tile, limit_ns, clear_words);
    } else {
        scan_u32_kernel<256, 2, INCLUSIVE, OP><<<n_tiles, 256, 0, stream>>>(data, n, total, carry_in, hdr, desc,
                                                                        n_tiles, head, skip_tile, limit_ns,
                                                                        clear_words);
    }
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

// Workspace bytes that serve a scan of any length from 1 to m (the
// one-tile-per-block kernel of lengths below the persistent threshold has
// more, smaller tiles).
size_t scan_workspace_bytes_upto(unsigned long long m) {
    const size_t a = scan_workspace_bytes(m);
    if (m < kPersistentMinN) return a;
    const size_t b = scan_workspace_bytes(kPersistentMinN - 1);
    return a > b ? a : b;
}

// One chunk of a longer add-scan: carry_in (device, or NULL for none) is
// the wrapped sum of everything before the chunk; total gets the carry-in
// plus the chunk's sum. total must not be carry_in: the block holding tile 0
// may read the carry-in after the last tile has written the total.
int scan_chunk_launch(bool inclusive, uint32_t *data, unsigned long long n, const uint32_t *carry_in,
                      uint32_t *total, void *ws, size_t ws_bytes, cudaStream_t stream) {
    return inclusive ? scan_launch<true>(data, n, total, ws, ws_bytes, stream, 0xffffffffu, kDefaultLimitNs, carry_in)
                     : scan_launch<false>(data, n, total, ws, ws_bytes, stream, 0xffffffffu, kDefaultLimitNs, carry_in);
}

// The inclusive form with its total, for the runs layout.
int scan_inclusive_launch(uint32_t *data, unsigned long long n, uint32_t *total, void *ws, size_t ws_bytes,
                          cudaStream_t stream) {
    return scan_launch<true>(data, n, total, ws, ws_bytes, stream, 0xffffffffu, kDefaultLimitNs);
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int scan_exclusive_u32(uint32_t *data, size_t n, uint32_t *total, void *ws, size_t ws_bytes,
                                  u32scan_stream_t stream) {
    return scan_launch<false>(data, n, total, ws, ws_bytes, (cudaStream_t)stream, 0xffffffffu, kDefaultLimitNs);
}

extern "C" int scan_inclusive_u32(uint32_t *data, size_t n, uint32_t *total, void *ws, size_t ws_bytes,
                                  u32scan_stream_t stream) {
    return scan_launch<true>(data, n, total, ws, ws_bytes, (cudaStream_t)stream, 0xffffffffu, kDefaultLimitNs);
}

extern "C" int scan_exclusive_u32_carry(uint32_t *data, size_t n, const uint32_t *carry_in, uint32_t *total,
                                        void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    if (n > 0 && total != nullptr && total == carry_in) return U32SCAN_EINVAL;
    if (reinterpret_cast<uintptr_t>(carry_in) & 3) return U32SCAN_EINVAL;
    return scan_chunk_launch(false, data, n, carry_in, total, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int scan_inclusive_u32_carry(uint32_t *data, size_t n, const uint32_t *carry_in, uint32_t *total,
                                        void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    if (n > 0 && total != nullptr && total == carry_in) return U32SCAN_EINVAL;
    if (reinterpret_cast<uintptr_t>(carry_in) & 3) return U32SCAN_EINVAL;
    return scan_chunk_launch(true, data, n, carry_in, total, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int scan_u32_op(int op, int inclusive, uint32_t *data, size_t n, uint32_t *total, void *ws,
                           size_t ws_bytes, u32scan_stream_t stream) {
    const cudaStream_t s = (cudaStream_t)stream;
    const unsigned int k = 0xffffffffu;
    const unsigned long long lim = kDefaultLimitNs;
#define U32SCAN_OP_CASE(CODE)                                                                 \
    case CODE:                                                                               \
        return inclusive ? scan_launch<true, CODE>(data, n, total, ws, ws_bytes, s, k, lim)  \
                         : scan_launch<false, CODE>(data, n, total, ws, ws_bytes, s, k, lim);
    switch (op) {
        U32SCAN_OP_CASE(kAdd)
        U32SCAN_OP_CASE(kMul)
        U32SCAN_OP_CASE(kAnd)
        U32SCAN_OP_CASE(kOr)
        U32SCAN_OP_CASE(kXor)
        U32SCAN_OP_CASE(kMin)
        U32SCAN_OP_CASE(kMax)
    default:
        return U32SCAN_EINVAL;
    }
#undef U32SCAN_OP_CASE
}

extern "C" int u32scan_test_scan_skip_publish(uint32_t *data, size_t n, uint32_t *total, void *ws, size_t ws_bytes,
                                              unsigned int skip_tile, unsigned long long limit_ns,
                                              u32scan_stream_t stream) {
    return scan_launch<false>(data, n, total, ws, ws_bytes, (cudaStream_t)stream, skip_tile, limit_ns);
}

// ---------------------------------------------------------------------------
// Allocation-free exclusive scan.
//
// Some callers cannot allocate device memory at all: code running where
// cudaMalloc is forbidden or unavailable (inside a custom allocator's own
// callbacks, a real-time path with a no-allocation rule, an embedding
// runtime that hands out only the buffers it owns). For them the carry
// workspace lives in a fixed file-scope device array, sized for n up to
// kStaticMaxN. Every GPU that loads this library holds the array (about
// 4 MiB) until the process exits.
//
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up once per device, with that device current, through
// cudaGetSymbolAddress. That lookup happens on the first call on each device;
// make that first call before any stream capture begins.
// ---------------------------------------------------------------------------
namespace u32scan {

constexpr unsigned long long kStaticMaxN = 1ull << 31;
// Header plus one carry word per tile for tiles as small as 4096 elements.
constexpr size_t kStaticScratchBytes = (kHeaderBytes + 8 * ((kStaticMaxN + 3) / 4096 + 2) + 255) / 256 * 256;

static __device__ __align__(256) unsigned char g_scan_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
static std::mutex g_static_mu;
static void *g_static_addr[kMaxDevices];

static int static_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return U32SCAN_ECUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scan_static_scratch) != cudaSuccess || p == nullptr) return U32SCAN_ECUDA;
        g_static_addr[dev] = p;
    }
    *out = g_static_addr[dev];
    return U32SCAN_OK;
}

// Sets the array's epoch (test hook below): one thread, on the stream.
__global__ void static_set_epoch_kernel(WsHeader *hdr, unsigned int epoch) { hdr->epoch = epoch; }

}  // namespace u32scan

extern "C" int scan_exclusive_u32_noalloc(uint32_t *data, size_t n, uint32_t *total, u32scan_stream_t stream) {
    if (n > kStaticMaxN) return U32SCAN_EINVAL;
    if (n == 0)
        return scan_launch<false>(data, 0, total, nullptr, 0, (cudaStream_t)stream, 0xffffffffu, kDefaultLimitNs);
    void *ws = nullptr;
    const int rc = static_scratch(&ws);
    if (rc != U32SCAN_OK) return rc;
    if (scan_workspace_bytes(n) > kStaticScratchBytes) return U32SCAN_EINVAL;
    // The array keeps the previous call's contents. Carry words are tagged
    // with a call counter, and the last block out of each launch resets the
    // tile counter and advances that call counter (also after a launch that
    // stopped early on a timeout), so nothing needs clearing between calls.
    return scan_launch<false>(data, n, total, ws, kStaticScratchBytes, (cudaStream_t)stream, 0xffffffffu,
                              kDefaultLimitNs);
}

extern "C" int u32scan_check_noalloc(u32scan_stream_t stream) {
    void *ws = nullptr;
    int rc = static_scratch(&ws);
    if (rc != U32SCAN_OK) return rc;
    rc = u32scan_check(ws, stream);
    if (rc == U32SCAN_ETIMEOUT) {
        // a launch that stopped early may have left the tile counter unreset:
        // start the array afresh (every caller's next call finds it zeroed)
        if (cudaMemsetAsync(ws, 0, kStaticScratchBytes, (cudaStream_t)stream) != cudaSuccess ||
            cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
            return U32SCAN_ECUDA;
    }
    return rc;
}

extern "C" int u32scan_test_noalloc_skip_publish(uint32_t *data, size_t n, uint32_t *total, unsigned int skip_tile,
                                                 unsigned long long limit_ns, u32scan_stream_t stream) {
    if (n > kStaticMaxN) return U32SCAN_EINVAL;
    void *ws = nullptr;
    const int rc = static_scratch(&ws);
    if (rc != U32SCAN_OK) return rc;
    return scan_launch<false>(data, n, total, ws, kStaticScratchBytes, (cudaStream_t)stream, skip_tile, limit_ns);
}

extern "C" int u32scan_test_noalloc_set_epoch(unsigned int epoch, u32scan_stream_t stream) {
    void *ws = nullptr;
    const int rc = static_scratch(&ws);
    if (rc != U32SCAN_OK) return rc;
    static_set_epoch_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(static_cast<WsHeader *>(ws), epoch);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

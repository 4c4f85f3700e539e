// scan64.cu -- exclusive and inclusive scans of u64 rows, in place, with
// the fold, under the integer operators of CAIRN's reduce and scan.
//
// Source: the CAIRN "Concurrency" page, "reduce and compact" (the operators
// add_wrap, mul_wrap, &, |, ^, min and max on integers; its examples reduce
// u64 terms) and "scan" (the operators are those of reduce; exclusive and
// inclusive forms; may run in place). add_wrap and mul_wrap wrap at 2^64.
//
// Kernels: for long rows a persistent block per SM (bulk-copy ring, one-
// tile software pipeline, bulk-copy stores, as scan.cu's long-row kernel);
// for short rows one tile per block. Tiles are drawn in order from the
// workspace counter (so every predecessor of a waiting tile is running), and
// carries pass by decoupled look-back. A carry is 64 bits, wider than the value
// field of the library's tagged carry word, so each tile publishes two
// tagged words, the low and the high half of its value, each in the u32
// scans' word format (value, P bit, epoch tag). A reader accepts a tile only
// when both words carry this call's tag and the same P bit: the two halves
// are then of one value (each word is written once per state and epoch), so
// relaxed loads suffice and a torn read is seen as "not ready yet".
//
// Layout inside a tile: warp w owns the w-th run of 64 * V elements; lane l
// holds, for r = 0 .. V-1, the two elements at 64 * r + 2 * l of that run
// (one 16-byte load and store each).
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

template <int OP>
struct Monoid64 {
    static __device__ __forceinline__ unsigned long long identity() {
        return OP == kMul ? 1ull : (OP == kAnd || OP == kMin) ? ~0ull : 0ull;
    }
    static __device__ __forceinline__ unsigned long long apply(unsigned long long a, unsigned long long b) {
        switch (OP) {
        case kAdd: return a + b;
        case kMul: return a * b;
        case kAnd: return a & b;
        case kOr: return a | b;
        case kXor: return a ^ b;
        case kMin: return a < b ? a : b;
        default: return a > b ? a : b;
        }
    }
    static __device__ __forceinline__ unsigned long long warp_fold(unsigned long long v) {
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) v = apply(v, __shfl_xor_sync(0xffffffffu, v, d));
        return v;
    }
    static __device__ __forceinline__ unsigned long long warp_inclusive(unsigned long long x, int lane) {
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x = apply(y, x);
        }
        return x;
    }
    static __device__ __forceinline__ unsigned long long warp_exclusive(unsigned long long inc,
                                                                       unsigned long long own, int lane) {
        if (OP == kAdd) return inc - own;
        const unsigned long long prev = __shfl_up_sync(0xffffffffu, inc, 1);
        return lane == 0 ? identity() : prev;
    }
};

// Carry words of tile t at desc2[2t] (low half) and desc2[2t + 1] (high).
__device__ __forceinline__ void publish64(unsigned long long *desc2, unsigned int t, unsigned long long v,
                                          bool inclusive, unsigned long long tag) {
    const unsigned long long f = tag | (inclusive ? kFlagP : 0ull);
    st_relaxed(desc2 + 2ull * t, f | (v & 0xffffffffull));
    st_relaxed(desc2 + 2ull * t + 1, f | (v >> 32));
}

// Fold (under OP) of tiles 0 .. t-1, by a warp: 32 tiles a round trip,
// lane l reading the tile l + 1 places back; stops at the nearest tile
// whose carry is an inclusive prefix.
// Lane l's word pair of the tile l + 1 places before tile t (a virtual
// inclusive prefix before tile 0): the walk's first window, which a caller
// may load early so that its round trip overlaps other work.
template <int OP>
__device__ __forceinline__ void window64(const unsigned long long *desc2, long long idx, unsigned long long tag,
                                         unsigned long long &lo, unsigned long long &hi) {
    using M = Monoid64<OP>;
    if (idx >= 0) {
        lo = ld_relaxed(desc2 + 2 * idx);
        hi = ld_relaxed(desc2 + 2 * idx + 1);
    } else {
        lo = tag | kFlagP | (M::identity() & 0xffffffffull);
        hi = tag | kFlagP | (M::identity() >> 32);
    }
}

template <int OP>
__device__ unsigned long long lookback64(const unsigned long long *desc2, unsigned int t, unsigned long long tag,
                                         WsHeader *hdr, unsigned long long limit_ns, int lane,
                                         unsigned long long lo, unsigned long long hi) {
    using M = Monoid64<OP>;
    if (t == 0) return M::identity();
    unsigned long long prefix = M::identity();
    long long pos = (long long)t - 1;
    auto load = [&](long long idx, unsigned long long &l, unsigned long long &h) { window64<OP>(desc2, idx, tag, l, h); };
    while (true) {
        unsigned long long t0 = 0;
        for (unsigned int iter = 0;; ++iter) {
            const bool ready = (lo & kTagMask) == tag && (hi & kTagMask) == tag && ((lo ^ hi) & kFlagP) == 0;
            const bool incl = ready && (lo & kFlagP);
            const unsigned int m = __ballot_sync(0xffffffffu, !ready || incl);
            const unsigned long long v = ((hi & 0xffffffffull) << 32) | (lo & 0xffffffffull);
            if (m == 0) {  // 32 aggregates: fold them and move back
                prefix = M::apply(prefix, M::warp_fold(v));
                break;
            }
            const int stop = __ffs(m) - 1;
            if (__shfl_sync(0xffffffffu, ready ? 1u : 0u, stop)) {  // an inclusive prefix, all nearer ready
                prefix = M::apply(prefix, M::warp_fold(lane <= stop ? v : M::identity()));
                return prefix;
            }
            if (iter == 0) t0 = __shfl_sync(0xffffffffu, globaltimer(), 0);
            if (iter >= 8) __nanosleep(32);
            if (!ready) load(pos - lane, lo, hi);
            const unsigned long long now = __shfl_sync(0xffffffffu, globaltimer(), 0);
            if (iter > 0 && (now - t0 > limit_ns || iter >= kMaxSpinIters)) {
                if (lane == 0) report_timeout(hdr, t);
                if (!ready) {  // give up: treat as the identity's inclusive prefix
                    lo = tag | kFlagP | (M::identity() & 0xffffffffull);
                    hi = tag | kFlagP | (M::identity() >> 32);
                }
            }
        }
        pos -= 32;
        load(pos - lane, lo, hi);
    }
}

template <int THREADS, int V, int MINB, bool INCLUSIVE, int OP>
__global__ void __launch_bounds__(THREADS, MINB)
scan_u64_kernel(unsigned long long *__restrict__ data, unsigned long long n, unsigned long long *total,
                WsHeader *hdr, unsigned long long *desc2, unsigned int n_tiles, unsigned int head,
                unsigned long long limit_ns, unsigned long long clear_words) {
    using M = Monoid64<OP>;
    constexpr int WARPS = THREADS / 32;
    constexpr unsigned long long TILE = (unsigned long long)THREADS * V * 2;
    static_assert(WARPS <= 32, "one warp scans the warp totals");
    __shared__ unsigned int s_tile, s_epoch;
    __shared__ unsigned long long s_warp[WARPS];

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

    const unsigned long long tile_v0 = (unsigned long long)t * TILE;
    const unsigned int li0 = (unsigned int)warp * (64 * V) + 2u * (unsigned int)lane;
    const unsigned int lo = tile_v0 < head ? (unsigned int)(head - tile_v0) : 0u;
    const unsigned long long left = head + n - tile_v0;
    const unsigned int hi = left < TILE ? (unsigned int)left : (unsigned int)TILE;
    const bool full = lo == 0 && hi == TILE;
    // The tile's virtual element 0 is 16-byte aligned; only elements in
    // [lo, hi) are dereferenced.
    unsigned long long *tbase =
        reinterpret_cast<unsigned long long *>(reinterpret_cast<uintptr_t>(data) - 8ull * head) + tile_v0;

    ulonglong2 x[V];
    if (full) {
#pragma unroll
        for (int r = 0; r < V; ++r) x[r] = __ldcs(reinterpret_cast<const ulonglong2 *>(tbase + li0 + 64 * r));
    } else {
#pragma unroll
        for (int r = 0; r < V; ++r) {
            const unsigned int a = li0 + 64 * r;
            x[r].x = (a >= lo && a < hi) ? tbase[a] : M::identity();
            x[r].y = (a + 1 >= lo && a + 1 < hi) ? tbase[a + 1] : M::identity();
        }
    }
    // per-round warp scans, carried from round to round
    unsigned long long carry = M::identity();
#pragma unroll
    for (int r = 0; r < V; ++r) {
        const unsigned long long sum = M::apply(x[r].x, x[r].y);
        const unsigned long long inc = M::warp_inclusive(sum, lane);
        const unsigned long long ex = M::apply(carry, M::warp_exclusive(inc, sum, lane));
        if (INCLUSIVE) {
            x[r].x = M::apply(ex, x[r].x);
            x[r].y = M::apply(x[r].x, x[r].y);
        } else {
            const unsigned long long a = x[r].x;
            x[r].x = ex;
            x[r].y = M::apply(ex, a);
        }
        carry = M::apply(carry, __shfl_sync(0xffffffffu, inc, 31));
    }
    if (lane == 0) s_warp[warp] = carry;
    __syncthreads();

    if (warp == 0) {
        const unsigned long long wt = lane < WARPS ? s_warp[lane] : M::identity();
        const unsigned long long winc = M::warp_inclusive(wt, lane);
        const unsigned long long agg = __shfl_sync(0xffffffffu, winc, 31);
        const unsigned long long wex = M::warp_exclusive(winc, wt, lane);
        if (lane == 0) publish64(desc2, t, agg, t == 0, tag);
        unsigned long long wlo, whi;
        window64<OP>(desc2, (long long)t - 1 - lane, tag, wlo, whi);
        const unsigned long long prefix = lookback64<OP>(desc2, t, tag, hdr, limit_ns, lane, wlo, whi);
        if (lane == 0 && t != 0) publish64(desc2, t, M::apply(prefix, agg), true, tag);
        if (lane < WARPS) s_warp[lane] = M::apply(prefix, wex);
        if (t == n_tiles - 1u && lane == 0 && total != nullptr) *total = M::apply(prefix, agg);
    }
    __syncthreads();

    const unsigned long long base = s_warp[warp];
#pragma unroll
    for (int r = 0; r < V; ++r) {
        x[r].x = M::apply(base, x[r].x);
        x[r].y = M::apply(base, x[r].y);
    }
    if (full) {
#pragma unroll
        for (int r = 0; r < V; ++r) __stcs(reinterpret_cast<ulonglong2 *>(tbase + li0 + 64 * r), x[r]);
    } else {
#pragma unroll
        for (int r = 0; r < V; ++r) {
            const unsigned int a = li0 + 64 * r;
            if (a >= lo && a < hi) tbase[a] = x[r].x;
            if (a + 1 >= lo && a + 1 < hi) tbase[a + 1] = x[r].y;
        }
    }
    finish_period(hdr, s_epoch, desc2, clear_words);
}

// Persistent form for long rows, the u64 counterpart of scan.cu's
// persistent kernel: each block loops over tiles drawn in order from the
// counter, keeping S tiles in flight as 1-D bulk copies into a ring of
// shared-memory stages, software-pipelined by one tile (it scans the next
// tile and publishes that tile's aggregate before walking the current
// tile's look-back), and stores full tiles with one 1-D bulk copy from an
// output buffer. Each block draws exactly S ids past the last tile; the
// last draw of the launch re-arms the header.
template <int THREADS, int V, int S, bool INCLUSIVE, int OP>
__global__ void __launch_bounds__(THREADS, 1)
scan_u64_persistent(unsigned long long *__restrict__ data, unsigned long long n, unsigned long long *total,
                    WsHeader *hdr, unsigned long long *desc2, unsigned int n_tiles, unsigned int head,
                    unsigned long long limit_ns, unsigned long long clear_words) {
    using M = Monoid64<OP>;
    constexpr int WARPS = THREADS / 32;
    constexpr unsigned int TILE = THREADS * V * 2;
    constexpr unsigned int TILE_BYTES = TILE * 8;
    constexpr unsigned int TILE_U4 = TILE_BYTES / 16;
    static_assert(WARPS <= 32, "one warp scans the warp totals");
    static_assert(S >= 2, "the pipeline reads one stage ahead");
    extern __shared__ __align__(128) ulonglong2 stage64[];  // S stages of TILE elements, then the output buffer
    __shared__ __align__(8) unsigned long long bar[S];
    __shared__ unsigned int s_tile[S];
    __shared__ unsigned long long s_wt[2][WARPS];
    __shared__ unsigned long long s_base[WARPS];
    __shared__ unsigned int s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned int last_draw = n_tiles + (unsigned int)S * gridDim.x - 1u;
    unsigned long long *vbase = reinterpret_cast<unsigned long long *>(reinterpret_cast<uintptr_t>(data) - 8ull * head);
    const bool producer = threadIdx.x == THREADS - 32;
    unsigned int latest_parity = 0;  // producer: bit st = phase parity of stage st's latest draw

    auto tile_full = [&](unsigned int id) {
        const unsigned long long v0 = (unsigned long long)id * TILE;
        return v0 >= head && v0 + TILE <= head + n;
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
            mbar_arrive_expect_tx(b, TILE_BYTES);
            bulk_load(smem_u32(stage64 + st * TILE_U4), vbase + (unsigned long long)id * TILE, TILE_BYTES, b);
        } else {
            mbar_arrive(b);  // nothing to copy: a partial tile reads global memory, a past-the-end draw stops
        }
    };
    const unsigned int li0 = (unsigned int)warp * (64 * V) + 2u * (unsigned int)lane;
    volatile unsigned int *vs_tile = s_tile;

    // Read draw u (stage u % S) into x and scan it per warp (warp totals to
    // s_wt[u & 1]); returns the tile, n_tiles past the end, n_tiles + 1 on a
    // timed-out copy.
    auto read_tile = [&](unsigned int u, ulonglong2 (&x)[V]) -> unsigned int {
        const int st = (int)(u % S);
        if (!mbar_wait_bounded(smem_u32(&bar[st]), (u / S) & 1u, limit_ns)) {
            report_timeout(hdr, 0xfffffffeu);
            return n_tiles + 1u;
        }
        const unsigned int t = vs_tile[st];
        if (t >= n_tiles) return n_tiles;
        if (tile_full(t)) {
            const ulonglong2 *sb = stage64 + st * TILE_U4 + (li0 >> 1);
#pragma unroll
            for (int r = 0; r < V; ++r) x[r] = sb[32 * r];
        } else {
            unsigned int lo, hi;
            tile_range(t, lo, hi);
            const unsigned long long *tb = vbase + (unsigned long long)t * TILE;
#pragma unroll
            for (int r = 0; r < V; ++r) {
                const unsigned int a = li0 + 64 * r;
                x[r].x = (a >= lo && a < hi) ? tb[a] : M::identity();
                x[r].y = (a + 1 >= lo && a + 1 < hi) ? tb[a + 1] : M::identity();
            }
        }
        unsigned long long carry = M::identity();
#pragma unroll
        for (int r = 0; r < V; ++r) {
            const unsigned long long sum = M::apply(x[r].x, x[r].y);
            const unsigned long long inc = M::warp_inclusive(sum, lane);
            const unsigned long long ex = M::apply(carry, M::warp_exclusive(inc, sum, lane));
            if (INCLUSIVE) {
                x[r].x = M::apply(ex, x[r].x);
                x[r].y = M::apply(x[r].x, x[r].y);
            } else {
                const unsigned long long a = x[r].x;
                x[r].x = ex;
                x[r].y = M::apply(ex, a);
            }
            carry = M::apply(carry, __shfl_sync(0xffffffffu, inc, 31));
        }
        if (lane == 0) s_wt[u & 1][warp] = carry;
        return t;
    };
    // Store the current tile: a full tile through the output buffer and one
    // bulk copy by thread 0 (whose previous copy finished reading the buffer
    // before barrier B), a partial tile element by element.
    auto store_tile = [&](unsigned int t, const ulonglong2 (&x)[V], unsigned long long base) {
        unsigned long long *tb = vbase + (unsigned long long)t * TILE;
        if (tile_full(t)) {
            ulonglong2 *ob = stage64 + S * TILE_U4;
#pragma unroll
            for (int r = 0; r < V; ++r) {
                ulonglong2 y;
                y.x = M::apply(base, x[r].x);
                y.y = M::apply(base, x[r].y);
                ob[(li0 >> 1) + 32 * r] = y;
            }
            fence_proxy_async_smem();
            __syncthreads();  // barrier C: the output buffer is complete
            if (threadIdx.x == 0) bulk_store(tb, smem_u32(ob), TILE_BYTES);
        } else {
            unsigned int lo, hi;
            tile_range(t, lo, hi);
#pragma unroll
            for (int r = 0; r < V; ++r) {
                const unsigned int a = li0 + 64 * r;
                if (a >= lo && a < hi) tb[a] = M::apply(base, x[r].x);
                if (a + 1 >= lo && a + 1 < hi) tb[a + 1] = M::apply(base, x[r].y);
            }
        }
    };
    auto block_aggregate = [&](int slot, unsigned long long &wex) -> unsigned long long {
        const unsigned long long wt = lane < WARPS ? s_wt[slot][lane] : M::identity();
        const unsigned long long winc = M::warp_inclusive(wt, lane);
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

    ulonglong2 xc[V], xn[V];
    unsigned int tc = read_tile(0, xc);
    unsigned long long agg_c = 0, wex_c = 0;
    if (!__syncthreads_or(tc >= n_tiles)) {
        if (producer) {
            fence_proxy_async_smem();
            issue(0);
            latest_parity ^= 1u;
        }
        if (warp == 0) {
            agg_c = block_aggregate(0, wex_c);
            if (lane == 0) publish64(desc2, tc, agg_c, tc == 0, tag);
        }
        for (unsigned int u = 1;; ++u) {
            const unsigned int tn = read_tile(u, xn);
            const bool more = !__syncthreads_or(tn >= n_tiles);  // barrier A
            unsigned long long agg_n = 0, wex_n = 0;
            if (more && producer) {
                fence_proxy_async_smem();
                const int st = (int)(u % S);
                issue(st);
                latest_parity ^= 1u << st;
            }
            if (warp == 0) {
                // the current tile's first window, loaded before the next
                // tile's aggregate so that its round trip overlaps that work
                unsigned long long wlo, whi;
                window64<OP>(desc2, (long long)tc - 1 - lane, tag, wlo, whi);
                if (more) {
                    agg_n = block_aggregate((int)(u & 1), wex_n);
                    if (lane == 0) publish64(desc2, tn, agg_n, tn == 0, tag);
                }
                const unsigned long long prefix = lookback64<OP>(desc2, tc, tag, hdr, limit_ns, lane, wlo, whi);
                if (lane == 0 && tc != 0) publish64(desc2, tc, M::apply(prefix, agg_c), true, tag);
                if (lane < WARPS) s_base[lane] = M::apply(prefix, wex_c);
                if (tc == n_tiles - 1u && lane == 0 && total != nullptr) *total = M::apply(prefix, agg_c);
            }
            if (threadIdx.x == 0) bulk_wait_read();  // output buffer free again
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
    if (producer) {
#pragma unroll
        for (int st = 0; st < S; ++st)
            (void)mbar_wait_bounded(smem_u32(&bar[st]), (latest_parity >> st) & 1u, limit_ns);
    }
    if (threadIdx.x == 0) bulk_wait_all();
    finish_period(hdr, s_epoch, desc2, clear_words);
}

// Shapes: short rows take one small tile per block (enough blocks to fill
// the GPU); long rows the persistent kernel. Chosen by measurement on
// GB300, overridable at build time for tuning sweeps.
#ifndef U32SCAN_S64_V
#define U32SCAN_S64_V 8
#endif
#ifndef U32SCAN_S64_STAGES
#define U32SCAN_S64_STAGES 2
#endif
constexpr int kS64T = 512, kS64V = U32SCAN_S64_V, kS64S = U32SCAN_S64_STAGES;
#ifndef U32SCAN_S64_MINN_LOG2
#define U32SCAN_S64_MINN_LOG2 20  // rows of at least 2^this elements take the persistent kernel
#endif
constexpr unsigned long long kScan64LargeMinN = 1ull << U32SCAN_S64_MINN_LOG2;
constexpr size_t kS64Smem = (size_t)(kS64S + 1) * kS64T * kS64V * 2 * 8;
static_assert(kS64Smem <= 227 * 1024, "shared memory");
struct Scan64Shape {
    int threads, v;
    unsigned long long tile() const { return (unsigned long long)threads * v * 2; }
};
static Scan64Shape scan64_shape(unsigned long long n) {
    return n >= kScan64LargeMinN ? Scan64Shape{kS64T, kS64V} : Scan64Shape{256, 2};
}

static std::mutex g_s64_mu;
static int g_s64_sms[64];
static int g_s64_bps[64][2][7];

template <bool INCLUSIVE, int OP>
static int scan64_grid(int *grid_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    std::lock_guard<std::mutex> lock(g_s64_mu);
    if (g_s64_sms[dev] == 0 &&
        cudaDeviceGetAttribute(&g_s64_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return U32SCAN_ECUDA;
    int &bps = g_s64_bps[dev][INCLUSIVE ? 1 : 0][OP];
    if (bps == 0) {
        auto kern = scan_u64_persistent<kS64T, kS64V, kS64S, INCLUSIVE, OP>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kS64Smem) != cudaSuccess)
            return U32SCAN_ECUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, kS64T, kS64Smem) != cudaSuccess || bps < 1)
            return U32SCAN_ECUDA;
    }
    *grid_out = g_s64_sms[dev] * bps;
    return U32SCAN_OK;
}

size_t scan64_workspace_bytes(unsigned long long n) {
    const unsigned long long tiles = (n + 1 + scan64_shape(n).tile() - 1) / scan64_shape(n).tile();
    return round_up(kHeaderBytes + 16 * tiles, 256);
}

// the fold of nothing: each operator's identity, copied to `total` when n = 0
static const unsigned long long kIdentity64[7] = {0ull, 1ull, ~0ull, 0ull, 0ull, ~0ull, 0ull};

template <bool INCLUSIVE, int OP>
static int scan64_launch(unsigned long long *data, unsigned long long n, unsigned long long *total, void *ws,
                         size_t ws_bytes, cudaStream_t stream) {
    if ((n > 0 && data == nullptr) || n >= (1ull << 32)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(data) & 7) || (reinterpret_cast<uintptr_t>(total) & 7)) return U32SCAN_EINVAL;
    if (n == 0) {
        if (total && cudaMemcpyAsync(total, &kIdentity64[OP], 8, cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return U32SCAN_ECUDA;
        return U32SCAN_OK;
    }
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < scan64_workspace_bytes(n))
        return U32SCAN_EWORKSPACE;
    const Scan64Shape sh = scan64_shape(n);
    const unsigned int head = (unsigned int)((reinterpret_cast<uintptr_t>(data) & 15) >> 3);
    const unsigned int n_tiles = (unsigned int)((n + head + sh.tile() - 1) / sh.tile());
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    unsigned long long *desc2 = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kHeaderBytes);
    const unsigned long long clear_words = tile_words_to_clear(ws_bytes);
    if (n >= kScan64LargeMinN) {
        int grid = 0;
        const int rc = scan64_grid<INCLUSIVE, OP>(&grid);
        if (rc != U32SCAN_OK) return rc;
        if ((unsigned int)grid > n_tiles) grid = (int)n_tiles;
        scan_u64_persistent<kS64T, kS64V, kS64S, INCLUSIVE, OP><<<grid, kS64T, kS64Smem, stream>>>(
            data, n, total, hdr, desc2, n_tiles, head, kDefaultLimitNs, clear_words);
    } else
        scan_u64_kernel<256, 2, 4, INCLUSIVE, OP><<<n_tiles, 256, 0, stream>>>(data, n, total, hdr, desc2, n_tiles,
                                                                            head, kDefaultLimitNs, clear_words);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int scan_u64_op(int op, int inclusive, uint64_t *data, size_t n, uint64_t *total, void *ws,
                           size_t ws_bytes, u32scan_stream_t stream) {
    const cudaStream_t s = (cudaStream_t)stream;
    unsigned long long *d = reinterpret_cast<unsigned long long *>(data);
    unsigned long long *t = reinterpret_cast<unsigned long long *>(total);
#define U32SCAN_OP64_CASE(CODE)                                                 \
    case CODE:                                                                 \
        return inclusive ? scan64_launch<true, CODE>(d, n, t, ws, ws_bytes, s) \
                         : scan64_launch<false, CODE>(d, n, t, ws, ws_bytes, s);
    switch (op) {
        U32SCAN_OP64_CASE(kAdd)
        U32SCAN_OP64_CASE(kMul)
        U32SCAN_OP64_CASE(kAnd)
        U32SCAN_OP64_CASE(kOr)
        U32SCAN_OP64_CASE(kXor)
        U32SCAN_OP64_CASE(kMin)
        U32SCAN_OP64_CASE(kMax)
    default:
        return U32SCAN_EINVAL;
    }
#undef U32SCAN_OP64_CASE
}

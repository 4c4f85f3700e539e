// compact_values.cu -- compaction of values: the kept values, in order, at
// the front of `out`, and their count.
//
// Source: the CAIRN "Concurrency" page, "reduce and compact": `compact out
// for i in n where p yield e` evaluates the test once per input, writes e
// for each selected i, in order, to the front of out (capacity n), returns
// how many it wrote, and leaves the rest of out unchanged. Here e is
// values[i] and the test is flags[i] != 0, or, with no flags, values[i] != 0
// (the page's `where xs[i] > 0` on unsigned values).
//
// Kernel: persistent, one block per SM, single pass with the look-back of
// the plain scan (scan.cu) over the keep indicator, the same two-stage
// bulk-copy pipeline as the index compaction (compact.cu) over the stream
// the keep bits come from (the flags, or the values themselves): a round
// reads the next tile's keep bits, counts them and publishes the count (its
// stage is re-armed at once), then walks the current tile's look-back,
// stages the tile's kept values at their tile-local rank in shared memory
// and stores them as one contiguous run. The values are read at the store,
// from L2: the values' own bulk copy put them there, or, with flags, the
// producer asks for an L2 prefetch of the tile's values when it starts the
// flags' copy; every warp loads them before warp 0's look-back, so the
// round trip overlaps it. Traffic: 4 bytes read per element (8 with flags),
// 4 written per kept element.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

template <int THREADS, int V, int S, bool FLAGS>
__global__ void __launch_bounds__(THREADS, 1)
compact_values_persistent(const uint32_t *__restrict__ values, const int32_t *__restrict__ flags,
                          unsigned long long n, uint32_t *__restrict__ out, int32_t *count, WsHeader *hdr,
                          unsigned long long *desc, unsigned int n_tiles, unsigned int head, int flags_aligned,
                          unsigned long long limit_ns, unsigned long long clear_words) {
    constexpr int WARPS = THREADS / 32;
    constexpr unsigned int CHUNK = 128 * V;
    constexpr unsigned int TILE = THREADS * V * 4;
    constexpr unsigned int TILE_BYTES = TILE * 4;
    static_assert(WARPS <= 32 && 4 * V <= 32, "one lane per warp; keep bits fit in a word");
    static_assert(S >= 2, "the pipeline reads one stage ahead");
    extern __shared__ __align__(128) uint4 smem_dyn[];  // S stages of the keep stream, then TILE staged values
    uint32_t *stage_out = reinterpret_cast<uint32_t *>(smem_dyn + S * (TILE / 4));
    __shared__ __align__(8) unsigned long long bar[S];
    __shared__ unsigned int s_tile[S];
    __shared__ unsigned int s_wt[2][WARPS];
    __shared__ unsigned int s_base[WARPS];
    __shared__ unsigned int s_prefix, s_kept, s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned int last_draw = n_tiles + (unsigned int)S * gridDim.x - 1u;
    const uint32_t *vvals = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(values) - 4ull * head);
    const int32_t *vflags = reinterpret_cast<const int32_t *>(reinterpret_cast<uintptr_t>(flags) - 4ull * head);
    // the stream the keep bits come from: flags, or the values themselves
    const uint4 *vkeep = FLAGS ? reinterpret_cast<const uint4 *>(vflags) : reinterpret_cast<const uint4 *>(vvals);
    const bool producer = threadIdx.x == THREADS - 32;
    unsigned int latest_parity = 0;  // bit st: parity of the latest phase armed on stage st

    auto tile_full = [&](unsigned int id) {
        const unsigned long long v0 = (unsigned long long)id * TILE;
        return v0 >= head && v0 + TILE <= head + n && (!FLAGS || flags_aligned);
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
            mbar_arrive_expect_tx(b, TILE_BYTES);
            bulk_load(smem_u32(smem_dyn + st * (TILE / 4)), vkeep + v0 / 4, TILE_BYTES, b);
            if (FLAGS) bulk_prefetch_l2(vvals + v0, TILE_BYTES);  // the values, read at the store
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
    const unsigned int li0 = (unsigned int)warp * CHUNK + 4u * (unsigned int)lane;
    volatile unsigned int *vs_tile = s_tile;

    // Read draw u's keep bits kb (bit 4r + c) and, per round, the kept count
    // before this lane's four elements within the warp (ex[r]); the warp's
    // count goes to s_wt[u & 1]. Draw u sits in stage u % S, phase u / S.
    auto read_tile = [&](unsigned int u, unsigned int &kb, unsigned int (&ex)[V]) -> unsigned int {
        const int st = (int)(u % S);
        if (!mbar_wait_bounded(smem_u32(&bar[st]), (u / S) & 1u, limit_ns)) {
            report_timeout(hdr, 0xfffffffeu);
            return n_tiles + 1u;
        }
        const unsigned int t = vs_tile[st];
        if (t >= n_tiles) return n_tiles;
        kb = 0;
        if (tile_full(t)) {
            const uint4 *sk = smem_dyn + st * (TILE / 4) + (li0 >> 2);
#pragma unroll
            for (int r = 0; r < V; ++r) {
                const uint4 f = sk[32 * r];
                kb |= ((f.x != 0) | ((f.y != 0) << 1) | ((f.z != 0) << 2) | ((f.w != 0) << 3)) << (4 * r);
            }
        } else {
            unsigned int lo, hi;
            tile_range(t, lo, hi);
            const unsigned long long v0 = (unsigned long long)t * TILE;
#pragma unroll
            for (int r = 0; r < V; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const unsigned int li = li0 + 128 * r + c;
                    if (li >= lo && li < hi && (FLAGS ? vflags[v0 + li] != 0 : vvals[v0 + li] != 0u))
                        kb |= 1u << (4 * r + c);
                }
        }
        unsigned int carry = 0;
#pragma unroll
        for (int r = 0; r < V; ++r) {
            const unsigned int pc = (unsigned int)__popc((kb >> (4 * r)) & 0xfu);
            const unsigned int inc = warp_inclusive_sum(pc, lane);
            ex[r] = carry + inc - pc;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_wt[u & 1][warp] = carry;
        return t;
    };
    auto block_aggregate = [&](int slot, unsigned int &wex) -> unsigned int {
        const unsigned int wt = lane < WARPS ? s_wt[slot][lane] : 0u;
        const unsigned int winc = warp_inclusive_sum(wt, lane);
        wex = winc - wt;
        return __shfl_sync(0xffffffffu, winc, 31);
    };

    unsigned int kbc = 0, kbn = 0;
    unsigned int exc[V], exn[V];
    unsigned int tc = read_tile(0, kbc, exc);
    unsigned int agg_c = 0, wex_c = 0;
    if (!__syncthreads_or(tc >= n_tiles)) {
        if (producer) {
            fence_proxy_async_smem();
            issue(0);
            latest_parity ^= 1u;
        }
        if (warp == 0) {
            agg_c = block_aggregate(0, wex_c);
            if (lane == 0) publish_aggregate(desc, tc, agg_c, tag);
        }
        for (unsigned int u = 1;; ++u) {
            const unsigned int tn = read_tile(u, kbn, exn);
            const bool more = !__syncthreads_or(tn >= n_tiles);  // barrier A
            if (more && producer) {
                fence_proxy_async_smem();
                const int st = (int)(u % S);
                issue(st);
                latest_parity ^= 1u << st;
            }
            // The current tile's values for its kept elements, from L2 (the
            // keep stream's bulk copy, or the producer's prefetch, brought
            // them there); loaded before the look-back so the round trip
            // overlaps it.
            const unsigned long long tile_v0 = (unsigned long long)tc * TILE;
            const bool full = tile_full(tc);
            uint4 xv[V];
#pragma unroll
            for (int r = 0; r < V; ++r) {
                const unsigned int b = (kbc >> (4 * r)) & 0xfu;
                xv[r] = make_uint4(0u, 0u, 0u, 0u);
                if (b == 0u) continue;
                if (full) {
                    xv[r] = __ldcg(reinterpret_cast<const uint4 *>(vvals + tile_v0 + li0 + 128 * r));
                } else {
                    const uint32_t *tb = vvals + tile_v0 + li0 + 128 * r;
                    if (b & 1u) xv[r].x = tb[0];
                    if (b & 2u) xv[r].y = tb[1];
                    if (b & 4u) xv[r].z = tb[2];
                    if (b & 8u) xv[r].w = tb[3];
                }
            }
            unsigned int agg_n = 0, wex_n = 0;
            if (warp == 0) {
                if (more) {
                    agg_n = block_aggregate((int)(u & 1u), wex_n);
                    if (lane == 0) publish_aggregate(desc, tn, agg_n, tag);
                }
                unsigned long long win[1];
                lookback_window<1>(desc, (long long)tc - 1, tag, lane, win);
                const unsigned int prefix = lookback_prefix_wide<1>(desc, tc, tag, hdr, limit_ns, lane, win);
                if (lane == 0 && tc != 0) publish_inclusive(desc, tc, prefix + agg_c, tag);
                if (lane < WARPS) s_base[lane] = wex_c;
                if (lane == 0) {
                    s_prefix = prefix;
                    s_kept = agg_c;
                    if (tc == n_tiles - 1u && count != nullptr) *count = (int32_t)(prefix + agg_c);
                }
            }
            __syncthreads();  // barrier B: the current tile's carries are visible
            {
                const unsigned int wbase = s_base[warp];
#pragma unroll
                for (int r = 0; r < V; ++r) {
                    const unsigned int b = (kbc >> (4 * r)) & 0xfu;
                    const unsigned int e[4] = {xv[r].x, xv[r].y, xv[r].z, xv[r].w};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if ((b >> c) & 1u) stage_out[wbase + exc[r] + __popc(b & ((1u << c) - 1u))] = e[c];
                }
            }
            __syncthreads();  // barrier C: the tile's kept values are staged
            {
                const unsigned int prefix = s_prefix, kept = s_kept;
                for (unsigned int j = threadIdx.x; j < kept; j += THREADS) __stcs(out + prefix + j, stage_out[j]);
            }
            if (!more) break;
            kbc = kbn;
#pragma unroll
            for (int r = 0; r < V; ++r) exc[r] = exn[r];
            tc = tn;
            agg_c = agg_n;
            wex_c = wex_n;
        }
    }
    // Leave no bulk copy in flight into this block's shared memory: wait
    // (bounded) for the latest phase armed on each stage (on the normal path
    // the outstanding draws are past the end, with nothing to copy).
    if (producer) {
#pragma unroll
        for (int st = 0; st < S; ++st)
            (void)mbar_wait_bounded(smem_u32(&bar[st]), (latest_parity >> st) & 1u, limit_ns);
    }
    finish_period(hdr, s_epoch, desc, clear_words);
}

// Launch shape, chosen by measurement on GB300 and overridable at build time
// for tuning sweeps: ring stages and u32x4 per lane.
#ifndef U32SCAN_CV_STAGES
#define U32SCAN_CV_STAGES 2
#endif
#ifndef U32SCAN_CV_V
#define U32SCAN_CV_V 8
#endif
constexpr int kVThreads = 512, kVStages = U32SCAN_CV_STAGES, kVV = U32SCAN_CV_V;
constexpr unsigned long long kVTile = (unsigned long long)kVThreads * kVV * 4;
constexpr size_t kVSmem = ((size_t)kVStages + 1) * kVTile * 4;
static_assert(kVSmem <= 227 * 1024, "shared memory");

size_t compact_values_workspace_bytes(unsigned long long n) {
    const unsigned long long tiles = (n + 3 + kVTile - 1) / kVTile;
    return round_up(kHeaderBytes + 8 * tiles, 256);
}

static std::mutex g_cv_mu;
static int g_cv_sms[64];
static bool g_cv_attr[64][2];

template <bool FLAGS>
static int compact_values_launch(const uint32_t *values, const int32_t *flags, unsigned long long n, uint32_t *out,
                                 int32_t *count, void *ws, size_t ws_bytes, cudaStream_t stream,
                                 unsigned long long limit_ns) {
    constexpr int V = kVV;
    constexpr unsigned long long TILE = kVTile;
    constexpr size_t SMEM = kVSmem;
    const unsigned int head = (unsigned int)((reinterpret_cast<uintptr_t>(values) & 15) >> 2);
    const int flags_aligned = ((reinterpret_cast<uintptr_t>(values) ^ reinterpret_cast<uintptr_t>(flags)) & 15) == 0;
    const unsigned int n_tiles = (unsigned int)((n + head + TILE - 1) / TILE);
    auto kern = compact_values_persistent<kVThreads, V, kVStages, FLAGS>;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    int sms;
    {
        std::lock_guard<std::mutex> lock(g_cv_mu);
        if (g_cv_sms[dev] == 0 &&
            cudaDeviceGetAttribute(&g_cv_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return U32SCAN_ECUDA;
        if (!g_cv_attr[dev][FLAGS ? 1 : 0]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) != cudaSuccess)
                return U32SCAN_ECUDA;
            g_cv_attr[dev][FLAGS ? 1 : 0] = true;
        }
        sms = g_cv_sms[dev];
    }
    const unsigned int grid = n_tiles < (unsigned int)sms ? n_tiles : (unsigned int)sms;
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    unsigned long long *desc = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kHeaderBytes);
    kern<<<grid, kVThreads, SMEM, stream>>>(values, flags, n, out, count, hdr, desc, n_tiles, head, flags_aligned,
                                           limit_ns, tile_words_to_clear(ws_bytes));
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int compact_values_u32(const uint32_t *values, const int32_t *flags, size_t n, uint32_t *out,
                                  int32_t *count, void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    const cudaStream_t s = (cudaStream_t)stream;
    if (n >= (1ull << 31)) return U32SCAN_EINVAL;
    if (n > 0 && (values == nullptr || out == nullptr)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(values) & 3) || (reinterpret_cast<uintptr_t>(flags) & 3) ||
        (reinterpret_cast<uintptr_t>(out) & 3) || (reinterpret_cast<uintptr_t>(count) & 3))
        return U32SCAN_EINVAL;
    if (n > 0) {  // out must not overlap the inputs: it is written while they are still read
        const uintptr_t o = reinterpret_cast<uintptr_t>(out), v = reinterpret_cast<uintptr_t>(values),
                        f = reinterpret_cast<uintptr_t>(flags), b = 4 * n;
        if ((o < v + b && v < o + b) || (flags && o < f + b && f < o + b)) return U32SCAN_EINVAL;
    }
    if (n == 0) {
        if (count && cudaMemsetAsync(count, 0, sizeof(int32_t), s) != cudaSuccess) return U32SCAN_ECUDA;
        return U32SCAN_OK;
    }
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < compact_values_workspace_bytes(n))
        return U32SCAN_EWORKSPACE;
    return flags ? compact_values_launch<true>(values, flags, n, out, count, ws, ws_bytes, s, kDefaultLimitNs)
                 : compact_values_launch<false>(values, nullptr, n, out, count, ws, ws_bytes, s, kDefaultLimitNs);
}

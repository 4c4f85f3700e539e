// compact.cu -- stream compaction: flags -> inclusive offsets -> gathered
// indices -> count.
//
// Source: the "parallel" package reference (entelechy docs), graph
// `compact` and its kernels: compact_blank fills every slot with -1,
// compact_offsets is an inclusive prefix sum (a kept element at i belongs at
// offsets[i] - 1), compact_total is the count as a row of one, and
// compact_gather scatters each kept index to its rank; a non-zero flag keeps
// its element. Also the CAIRN "Concurrency" page, "reduce and compact": the
// kept elements land in order at the front.
//
// The page's four kernels (blank, prefix, reduce, scatter with max) become
// one single-pass kernel here: every slot of `indices` is written exactly
// once, either with a kept index (the front [0, count)) or with -1 (the tail
// [count, n)), so the blank pass and the scatter's max rule disappear. The
// non-kept element with r non-kept elements before it writes -1 to slot
// n - 1 - r, which fills the tail without knowing the count first. Traffic:
// 4 bytes read and 8 written per element (flags; offsets and one slot).
//
// Kernel: persistent, one block per SM, the one-tile software pipeline of
// the plain scan (scan.cu) over the keep indicator (flag != 0): a 1-D bulk
// copy per tile of flags into a ring of shared-memory stages; each round
// reads and counts the next tile and publishes its kept count, then walks
// the current tile's look-back, writes its offsets with 16-byte stores, and
// writes its run of kept indices (staged in shared memory at their tile-
// local rank, then stored contiguously) and its run of -1 slots.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

#ifndef U32SCAN_C_V
#define U32SCAN_C_V 8
#endif
#ifndef U32SCAN_C_STAGES
#define U32SCAN_C_STAGES 2
#endif

namespace u32scan {

template <int THREADS, int V, int S>
__global__ void __launch_bounds__(THREADS, 1)
compact_persistent(const int32_t *__restrict__ flags, unsigned long long n, int32_t *offsets,
                   int32_t *__restrict__ indices, int32_t *count, WsHeader *hdr, unsigned long long *desc,
                   unsigned int n_tiles, unsigned int head, int offsets_aligned, unsigned long long limit_ns,
                   unsigned long long clear_words, const int32_t *kept_before, const int32_t *first_index) {
    constexpr int WARPS = THREADS / 32;
    constexpr unsigned int CHUNK = 128 * V;
    constexpr unsigned int TILE = THREADS * V * 4;
    constexpr unsigned int TILE_BYTES = TILE * 4;
    static_assert(WARPS <= 32 && 4 * V <= 32, "one lane per warp; keep bits fit in a word");
    extern __shared__ __align__(128) uint4 smem_dyn[];  // S stages of TILE flags, then TILE staged indices
    int32_t *stage_idx = reinterpret_cast<int32_t *>(smem_dyn + S * (TILE / 4));
    __shared__ __align__(8) unsigned long long bar[S];
    __shared__ unsigned int s_tile[S];
    __shared__ unsigned int s_wt[2][WARPS];
    __shared__ unsigned int s_base[WARPS];  // kept before warp w of the current tile (tile-local)
    __shared__ unsigned int s_prefix;       // kept before the current tile
    __shared__ unsigned int s_kept;         // kept in the current tile
    __shared__ unsigned int s_kbase, s_ibase;  // carry-ins: kept elements and elements before the array
    __shared__ unsigned int s_epoch;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const unsigned int last_draw = n_tiles + (unsigned int)S * gridDim.x - 1u;
    const int32_t *vflags = reinterpret_cast<const int32_t *>(reinterpret_cast<uintptr_t>(flags) - 4ull * head);
    int32_t *voffsets = reinterpret_cast<int32_t *>(reinterpret_cast<uintptr_t>(offsets) - 4ull * head);
    const bool producer = threadIdx.x == THREADS - 32;
    unsigned int latest_parity = 0;

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
            bulk_load(smem_u32(smem_dyn + st * (TILE / 4)), vflags + (unsigned long long)id * TILE, TILE_BYTES, b);
        } else {
            mbar_arrive(b);
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
    if (threadIdx.x == 0) {  // the array as one piece of a longer one: what lies before it
        s_kbase = kept_before ? (unsigned int)*kept_before : 0u;
        s_ibase = first_index ? (unsigned int)*first_index : 0u;
    }
    __syncthreads();
    const unsigned long long tag = tag_of(s_epoch);
    const unsigned int kbase = s_kbase, ibase = s_ibase;
    const unsigned int li0 = (unsigned int)warp * CHUNK + 4u * (unsigned int)lane;
    volatile unsigned int *vs_tile = s_tile;

    // Read draw u: keep bits kb (bit 4r + c) and, per round, the kept count
    // before this lane's four elements within the warp (ex[r]). The warp's
    // kept count goes to s_wt[u & 1].
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
            const int4 *sf = reinterpret_cast<const int4 *>(smem_dyn + st * (TILE / 4)) + (li0 >> 2);
#pragma unroll
            for (int r = 0; r < V; ++r) {
                const int4 f = sf[32 * r];
                kb |= ((f.x != 0) | ((f.y != 0) << 1) | ((f.z != 0) << 2) | ((f.w != 0) << 3)) << (4 * r);
            }
        } else {
            unsigned int lo, hi;
            tile_range(t, lo, hi);
            const int32_t *tf = vflags + (unsigned long long)t * TILE;
#pragma unroll
            for (int r = 0; r < V; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const unsigned int li = li0 + 128 * r + c;
                    if (li >= lo && li < hi && tf[li] != 0) kb |= 1u << (4 * r + c);
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


    unsigned int kbc = 0, kbn = 0;
    unsigned int exc[V], exn[V];
    unsigned int tc = read_tile(0, kbc, exc);
    unsigned int agg_c = 0, wex_c = 0;
    auto block_aggregate = [&](int slot, unsigned int &wex) -> unsigned int {
        const unsigned int wt = lane < WARPS ? s_wt[slot][lane] : 0u;
        const unsigned int winc = warp_inclusive_sum(wt, lane);
        wex = winc - wt;
        return __shfl_sync(0xffffffffu, winc, 31);
    };
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
            unsigned int agg_n = 0, wex_n = 0;
            if (more && producer) {
                fence_proxy_async_smem();
                const int st = (int)(u % S);
                issue(st);
                latest_parity ^= 1u << st;
            }
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

            // ---- store the current tile ----
            {
                const unsigned long long tile_v0 = (unsigned long long)tc * TILE;
                unsigned int lo, hi;
                tile_range(tc, lo, hi);
                const unsigned int prefix = s_prefix;
                const unsigned int kept = s_kept;
                const unsigned int wbase = s_base[warp];
                const long long e0 = (long long)tile_v0 - (long long)head;  // element index of tile slot 0
                if (offsets != nullptr) {
                    int32_t *to = voffsets + tile_v0;
                    const bool vec = offsets_aligned && tile_full(tc);
#pragma unroll
                    for (int r = 0; r < V; ++r) {
                        const unsigned int b = (kbc >> (4 * r)) & 0xfu;
                        const unsigned int o = kbase + prefix + wbase + exc[r];
                        const int4 y = make_int4((int)(o + (b & 1u)), (int)(o + __popc(b & 3u)),
                                                 (int)(o + __popc(b & 7u)), (int)(o + __popc(b)));
                        if (vec) {
                            __stcs(reinterpret_cast<int4 *>(to + li0 + 128 * r), y);
                        } else {
                            const int yy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const unsigned int li = li0 + 128 * r + c;
                                if (li >= lo && li < hi) to[li] = yy[c];
                            }
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < V; ++r) {
                    const unsigned int b = (kbc >> (4 * r)) & 0xfu;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if ((b >> c) & 1u)
                            stage_idx[wbase + exc[r] + __popc(b & ((1u << c) - 1u))] =
                                (int32_t)(ibase + e0 + li0 + 128 * r + c);
                }
                __syncthreads();  // barrier C: the tile's kept indices are staged
                for (unsigned int j = threadIdx.x; j < kept; j += THREADS) __stcs(indices + prefix + j, stage_idx[j]);
                // the tile's non-kept elements fill a run of the tail with -1
                const unsigned long long first = e0 < 0 ? 0ull : (unsigned long long)e0 + lo;
                const unsigned long long valid = hi - lo;
                const unsigned long long nk_before = first - prefix;  // non-kept elements before the tile
                const unsigned long long nk = valid - kept;
                int32_t *tail = indices + (n - nk_before - nk);
                for (unsigned int j = threadIdx.x; j < nk; j += THREADS) __stcs(tail + j, -1);
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
    if (producer) {
#pragma unroll
        for (int st = 0; st < S; ++st)
            (void)mbar_wait_bounded(smem_u32(&bar[st]), (latest_parity >> st) & 1u, limit_ns);
    }
    finish_period(hdr, s_epoch, desc, clear_words);
}

constexpr int kCThreads = 512, kCV = U32SCAN_C_V, kCStages = U32SCAN_C_STAGES;
constexpr unsigned long long kCTile = (unsigned long long)kCThreads * kCV * 4;
constexpr size_t kCSmem = (size_t)(kCStages + 1) * kCTile * 4;

size_t compact_workspace_bytes(unsigned long long n) {
    const unsigned long long tiles = (n + 3 + kCTile - 1) / kCTile;
    return round_up(kHeaderBytes + 8 * tiles, 256);
}

static std::mutex g_cmp_mu;
static int g_cmp_sms[64];
static bool g_cmp_attr[64];

static int compact_launch(const int32_t *flags, unsigned long long n, int32_t *offsets, int32_t *indices,
                          int32_t *count, void *ws, size_t ws_bytes, cudaStream_t stream,
                          unsigned long long limit_ns, const int32_t *kept_before = nullptr,
                          const int32_t *first_index = nullptr) {
    if (n >= (1ull << 31)) return U32SCAN_EINVAL;
    if (n > 0 && (flags == nullptr || indices == nullptr)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(flags) & 3) || (reinterpret_cast<uintptr_t>(offsets) & 3) ||
        (reinterpret_cast<uintptr_t>(indices) & 3) || (reinterpret_cast<uintptr_t>(count) & 3) ||
        (reinterpret_cast<uintptr_t>(kept_before) & 3) || (reinterpret_cast<uintptr_t>(first_index) & 3))
        return U32SCAN_EINVAL;
    if (n == 0) {
        if (count && cudaMemsetAsync(count, 0, sizeof(int32_t), stream) != cudaSuccess) return U32SCAN_ECUDA;
        return U32SCAN_OK;
    }
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < compact_workspace_bytes(n))
        return U32SCAN_EWORKSPACE;
    const unsigned int head = (unsigned int)((reinterpret_cast<uintptr_t>(flags) & 15) >> 2);
    const int offsets_aligned = ((reinterpret_cast<uintptr_t>(flags) ^ reinterpret_cast<uintptr_t>(offsets)) & 15) == 0;
    const unsigned int n_tiles = (unsigned int)((n + head + kCTile - 1) / kCTile);
    auto kern = compact_persistent<kCThreads, kCV, kCStages>;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    int sms;
    {
        std::lock_guard<std::mutex> lock(g_cmp_mu);
        if (g_cmp_sms[dev] == 0 &&
            cudaDeviceGetAttribute(&g_cmp_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return U32SCAN_ECUDA;
        if (!g_cmp_attr[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCSmem) != cudaSuccess)
                return U32SCAN_ECUDA;
            g_cmp_attr[dev] = true;
        }
        sms = g_cmp_sms[dev];
    }
    const unsigned int grid = n_tiles < (unsigned int)sms ? n_tiles : (unsigned int)sms;
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    unsigned long long *desc = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kHeaderBytes);
    kern<<<grid, kCThreads, kCSmem, stream>>>(flags, n, offsets, indices, count, hdr, desc, n_tiles, head,
                                             offsets_aligned, limit_ns, tile_words_to_clear(ws_bytes), kept_before,
                                             first_index);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int compact_indices_u32(const int32_t *flags, size_t n, int32_t *offsets, int32_t *indices,
                                   int32_t *count, void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    return compact_launch(flags, n, offsets, indices, count, ws, ws_bytes, (cudaStream_t)stream, kDefaultLimitNs);
}

extern "C" int compact_indices_u32_carry(const int32_t *flags, size_t n, const int32_t *kept_before,
                                         const int32_t *first_index, int32_t *offsets, int32_t *indices,
                                         int32_t *count, void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    return compact_launch(flags, n, offsets, indices, count, ws, ws_bytes, (cudaStream_t)stream, kDefaultLimitNs,
                          kept_before, first_index);
}

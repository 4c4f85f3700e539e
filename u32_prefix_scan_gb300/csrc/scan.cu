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

namespace u32scan {

template <int THREADS, int V, bool INCLUSIVE>
__global__ void __launch_bounds__(THREADS, (THREADS >= 512 ? 2 : 4))
scan_u32_kernel(uint32_t *__restrict__ data, unsigned long long n, uint32_t *total, WsHeader *hdr,
                unsigned long long *desc, unsigned int n_tiles, unsigned int head, unsigned int skip_tile,
                unsigned long long limit_ns) {
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
                e[c] = (li >= lo && li < hi) ? tbase[li] : 0u;
            }
            x[r] = make_uint4(e[0], e[1], e[2], e[3]);
        }
    }

    // Warp-level scan, r-major; x becomes the scan relative to the warp start.
    unsigned int carry = 0;
#pragma unroll
    for (int r = 0; r < V; ++r) {
        const unsigned int s = x[r].x + x[r].y + x[r].z + x[r].w;
        const unsigned int inc = warp_inclusive_sum(s, lane);
        const unsigned int ex = carry + (inc - s);
        if (INCLUSIVE) {
            x[r].x += ex;
            x[r].y += x[r].x;
            x[r].z += x[r].y;
            x[r].w += x[r].z;
        } else {
            const unsigned int a = x[r].x, b = x[r].y, c = x[r].z;
            x[r].x = ex;
            x[r].y = ex + a;
            x[r].z = x[r].y + b;
            x[r].w = x[r].z + c;
        }
        carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) s_warp[warp] = carry;
    __syncthreads();

    if (warp == 0) {
        const unsigned int wt = lane < WARPS ? s_warp[lane] : 0u;
        const unsigned int winc = warp_inclusive_sum(wt, lane);
        const unsigned int agg = __shfl_sync(0xffffffffu, winc, 31);
        const unsigned int prefix = lookback_sum(desc, t, agg, tag, hdr, limit_ns, t != skip_tile, lane);
        if (lane < WARPS) s_warp[lane] = prefix + (winc - wt);
        if (t == n_tiles - 1u && lane == 0 && total != nullptr) *total = prefix + agg;
    }
    __syncthreads();

    const unsigned int base = s_warp[warp];
#pragma unroll
    for (int r = 0; r < V; ++r) {
        x[r].x += base;
        x[r].y += base;
        x[r].z += base;
        x[r].w += base;
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
}

// Launch shapes, chosen by n: long arrays take wide tiles (few carries to
// chain), short ones narrow tiles (enough blocks to fill the GPU).
struct ScanShape {
    int threads, v;
    unsigned long long tile() const { return (unsigned long long)threads * v * 4; }
};

static ScanShape scan_shape(unsigned long long n) {
    if (n >= (1ull << 22)) return {512, 8};
    return {256, 2};
}

size_t scan_workspace_bytes(unsigned long long n) {
    const unsigned long long tiles = (n + 3 + scan_shape(n).tile() - 1) / scan_shape(n).tile();
    return round_up(kHeaderBytes + 8 * tiles, 256);
}

template <bool INCLUSIVE>
static int scan_launch(uint32_t *data, unsigned long long n, uint32_t *total, void *ws, size_t ws_bytes,
                       cudaStream_t stream, unsigned int skip_tile, unsigned long long limit_ns) {
    if ((n > 0 && data == nullptr) || n >= (1ull << 32)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(data) & 3) || (reinterpret_cast<uintptr_t>(total) & 3))
        return U32SCAN_EINVAL;
    if (n == 0) {
        if (total && cudaMemsetAsync(total, 0, sizeof(uint32_t), stream) != cudaSuccess) return U32SCAN_ECUDA;
        return U32SCAN_OK;
    }
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < scan_workspace_bytes(n))
        return U32SCAN_EWORKSPACE;
    const ScanShape sh = scan_shape(n);
    const unsigned int head = (unsigned int)((reinterpret_cast<uintptr_t>(data) & 15) >> 2);
    const unsigned int n_tiles = (unsigned int)((n + head + sh.tile() - 1) / sh.tile());
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    unsigned long long *desc = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kHeaderBytes);
    if (sh.threads == 512)
        scan_u32_kernel<512, 8, INCLUSIVE><<<n_tiles, 512, 0, stream>>>(data, n, total, hdr, desc, n_tiles, head,
                                                                        skip_tile, limit_ns);
    else
        scan_u32_kernel<256, 2, INCLUSIVE><<<n_tiles, 256, 0, stream>>>(data, n, total, hdr, desc, n_tiles, head,
                                                                        skip_tile, limit_ns);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
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
    // with a call counter, so stale ones are never taken for current ones;
    // only the tile counter must read zero when a launch starts. Each launch
    // leaves it at zero, and it is cleared here as well, in case an earlier
    // launch on this array never completed.
    if (cudaMemsetAsync(ws, 0, sizeof(unsigned int), (cudaStream_t)stream) != cudaSuccess) return U32SCAN_ECUDA;
    return scan_launch<false>(data, n, total, ws, kStaticScratchBytes, (cudaStream_t)stream, 0xffffffffu,
                              kDefaultLimitNs);
}

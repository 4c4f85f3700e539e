// runs.cu -- the runs layout of per-owner entry counts, and the owner of
// every entry.
//
// Source: the "parallel" package reference (entelechy docs), graph `runs`
// and its kernels: runs_ends is an inclusive prefix sum of the counts (owner
// i's run covers ends[i] - counts[i] up to, not including, ends[i]),
// runs_entries is the number of entries as a row of one, at least one so the
// row is never empty, and runs_slots is the row of `entries` slots, every
// one -1 until a scatter fills it. The function owner(e, ends) gives the
// owner of entry e from the ends.
//
// runs_layout_u32 is the library's inclusive scan (scan.cu), in place, with
// its total written to `entries`, then one fill kernel that raises the total
// to at least one and writes the -1 slots (4 bytes per slot, 16-byte
// stores).
//
// runs_owner_u32 evaluates owner(e, ends) for every entry at once, as a
// merge of the sorted row `ends` with the entry indices 0, 1, 2, ...: along
// this "merge path" owner i stands at position min(ends[i], E) + i (after
// the entries its run ends above and the owners before it; E = entries
// written), so the first p positions hold split(p) = #{i : min(ends[i], E)
// + i < p} owners, and an entry reached after i owners belongs to owner i.
// Persistent warps take equal slices of the path -- owners plus entries, so
// empty owners and long runs cost alike -- each finds its start by one
// warp-wide search in global memory, then walks its slice in tiles of 508
// positions with no block-wide barrier. A tile tests its owners 32 at a
// time (loaded while the previous tile was stored, as many chunks as that
// tile needed plus one, more on demand) until one chunk holds an owner the
// tile does not pass; each passed owner that ends a run of equal offsets
// marks the count of owners passed so far at its end's offset in shared
// memory; a warp max-scan turns the marks into every entry's owner, and each
// lane writes its 16 owners from registers with 16-byte stores, in a frame
// aligned to the owner row. Traffic: 4 bytes read per owner and 4 written
// per entry.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

#ifndef U32SCAN_RO_WARPS
#define U32SCAN_RO_WARPS 16
#endif
#ifndef U32SCAN_RO_VT
#define U32SCAN_RO_VT 16
#endif
#ifndef U32SCAN_RO_MINB
#define U32SCAN_RO_MINB 2
#endif
constexpr int kROWarps = U32SCAN_RO_WARPS, kROVT = U32SCAN_RO_VT, kROThreads = kROWarps * 32;
constexpr int kFillThreads = 256;

// The second step of the layout: entries = max(total, 1), then slots[0,
// min(entries, cap)) = -1. Every block reads the scan's total; block 0 may
// raise a zero total to one, which leaves every reader's max(total, 1) the
// same (relaxed accesses, so the concurrent read and write are well defined).
__global__ void __launch_bounds__(kFillThreads) runs_entries_slots_kernel(unsigned int *entries, int32_t *slots,
                                                                        unsigned long long cap) {
    const unsigned int total = ld_relaxed_u32(entries);
    const unsigned int e = total ? total : 1u;
    if (blockIdx.x == 0 && threadIdx.x == 0 && total == 0) st_relaxed_u32(entries, 1u);
    if (slots == nullptr) return;
    const unsigned long long m = e < cap ? e : cap;
    const unsigned long long tid = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    unsigned long long head = ((16u - (reinterpret_cast<uintptr_t>(slots) & 15u)) & 15u) >> 2;  // to a 16-byte boundary
    if (head > m) head = m;
    if (tid < head) slots[tid] = -1;
    const unsigned long long body = (m - head) >> 2;
    int4 *v = reinterpret_cast<int4 *>(slots + head);
    for (unsigned long long k = tid; k < body; k += stride) v[k] = make_int4(-1, -1, -1, -1);
    const unsigned long long done = head + 4 * body;
    if (tid < m - done) slots[done + tid] = -1;
}

// g(i) = min(ends[i], E) + i, owner i's position on the merge path.
__device__ __forceinline__ unsigned long long path_pos(const unsigned int *ends, unsigned long long i,
                                                       unsigned long long E) {
    const unsigned long long v = __ldg(ends + i);
    return (v < E ? v : E) + i;
}

// One warp: the least i in [lo, hi] with i == hi or g(i) >= d (g is
// non-decreasing, so the predicate is monotone). 32 probes a round shrink
// the range 32-fold; only indices below hi are read.
__device__ unsigned long long split_global(const unsigned int *ends, unsigned long long lo, unsigned long long hi,
                                           unsigned long long d, unsigned long long E, int lane) {
    while (hi - lo > 32) {
        const unsigned long long step = (hi - lo + 31) >> 5;
        const unsigned long long p = lo + (unsigned long long)(lane + 1) * step - 1;
        const bool pr = p >= hi || path_pos(ends, p, E) >= d;
        const unsigned int b = __ballot_sync(0xffffffffu, pr);
        if (b == 0) return hi;
        const int k = __ffs(b) - 1;
        const unsigned long long pk = lo + (unsigned long long)(k + 1) * step - 1;
        lo = lo + (unsigned long long)k * step;  // one past the last probe that failed
        if (pk < hi) hi = pk;
    }
    if (lo == hi) return lo;
    const unsigned long long p = lo + lane;
    const bool pr = p >= hi || path_pos(ends, p, E) >= d;
    const unsigned int b = __ballot_sync(0xffffffffu, pr);
    return b ? lo + (unsigned long long)(__ffs(b) - 1) : hi;
}

// owner[e] for e in [0, min(total, cap)), total = ends[n-1] > 0, n >= 1;
// the empty layout (total 0) writes its one slot, -1.
//
// Every warp walks its own slice of the path in tiles of 32 * VT positions,
// with no block-wide barriers. A tile starts after i0 owners and j0
// entries; owner k of the tile (global i0 + k) has rel_k = min(ends, E) - j0
// of the tile's entries before it and is passed inside the tile iff
// rel_k + k < q1 (the tile's length), a prefix of its owners since rel_k + k
// increases with k. The owner of tile entry jl is i0 + #{passed k : rel_k <=
// jl}: the last passed owner of each distinct rel_k (a unique writer, told
// by its neighbour's rel, which a shuffle brings) marks k + 1 at rel_k, a
// warp max-scan of the marks gives every entry's owner, and the owner at the
// passed/not-passed boundary gives the tile's count. Shared memory is
// indexed with one pad word per 32 so that the blocked scan is free of bank
// conflicts.
template <int WARPS, int VT>
__global__ void __launch_bounds__(WARPS * 32, U32SCAN_RO_MINB) runs_owner_kernel(const unsigned int *__restrict__ ends,
                                                                unsigned int n, int32_t *__restrict__ owner,
                                                                unsigned long long cap) {
    constexpr unsigned int Dw = 32u * VT;
    constexpr unsigned int TP = Dw - 4;  // path positions a tile: its entries fit the aligned frame
    constexpr unsigned int PADDED = Dw + Dw / 32;
    static_assert(VT % 4 == 0 && 32 % VT == 0, "a lane's frame positions: whole 16-byte stores, one pad");
    // marks, then the tile's owners; zero between tiles
    __shared__ unsigned int s_buf[WARPS][PADDED];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned int *buf = s_buf[warp];
    auto pad = [](unsigned int p) { return p + (p >> 5); };

    const unsigned int total = __ldg(ends + n - 1);
    if (total == 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && cap > 0) owner[0] = -1;
        return;
    }
    const unsigned int E = total < cap ? total : (unsigned int)cap;
    if (E == 0) return;
    const unsigned long long L = (unsigned long long)n + E;
    const unsigned long long tiles = (L + TP - 1) / TP;
    const unsigned long long nwarps = (unsigned long long)gridDim.x * WARPS;
    const unsigned long long per = (tiles + nwarps - 1) / nwarps;
    unsigned long long d0 = ((unsigned long long)blockIdx.x * WARPS + warp) * per * TP;
    if (d0 >= L) return;
    const unsigned long long d_end = d0 + per * TP < L ? d0 + per * TP : L;
    const unsigned int oa = (unsigned int)((reinterpret_cast<uintptr_t>(owner) >> 2) & 3u);  // owner's phase mod 16 B
    unsigned int i0 = (unsigned int)split_global(ends, d0 > E ? d0 - E : 0, d0 < n ? d0 : n, d0, E, lane);
#pragma unroll
    for (unsigned int p = lane; p < PADDED; p += 32) buf[p] = 0u;
    __syncwarp();
    unsigned int raw[VT];  // end values of the tile's first chunks, loaded ahead
    int loaded = 0;        // chunks of the current tile in raw (warp-uniform)

    while (d0 < d_end) {
        const unsigned int j0 = (unsigned int)(d0 - i0);  // entries before the tile, <= E
        const unsigned int q1 = (unsigned int)(d_end - d0 < TP ? d_end - d0 : TP);
        const unsigned int cnt = n - i0 < q1 ? n - i0 : q1;  // owners the tile can pass
        // Marks and owners live in a frame aligned to 16 bytes of the owner
        // row: tile entry jl sits at frame position jl + s_al.
        const unsigned int s_al = (oa + j0) & 3u;
        // Chunks of 32 owners: the ones loaded ahead (while the previous
        // tile stored), then more on demand until a chunk holds an owner the
        // tile does not pass (the passed owners are a prefix).
        unsigned int pass = 0u;
        int used = 0;
#pragma unroll
        for (int m = 0; m < VT; ++m) {
            if (32u * m >= cnt) break;
            const unsigned int k = (unsigned int)lane + 32u * m;
            if (m >= loaded) raw[m] = k < cnt ? __ldg(ends + i0 + k) : 0xffffffffu;  // warp-uniform test
            const unsigned int c = raw[m] < E ? raw[m] : E;
            const unsigned int r = c > j0 ? (c - j0 < Dw ? c - j0 : Dw) : 0u;
            const bool passed = k < cnt && r + k < q1;
            // the last passed owner of each run of equal offsets in the chunk
            // marks; a run crossing into the next chunk is settled by max
            const unsigned int rn = __shfl_down_sync(0xffffffffu, r, 1);
            const bool pn = __shfl_down_sync(0xffffffffu, passed ? 1u : 0u, 1) != 0u;
            if (passed && (lane == 31 || !pn || rn != r)) atomicMax(&buf[pad(r + s_al)], k + 1);
            if (passed) pass = k + 1;
            used = m + 1;
            if (__ballot_sync(0xffffffffu, passed) != 0xffffffffu) break;
        }
        // owners passed in the tile, held to what the entries left allow
        const unsigned int left = E - j0;
        const unsigned int lo1 = q1 > left ? q1 - left : 0u;
        unsigned int il1 = __reduce_max_sync(0xffffffffu, pass);
        il1 = il1 < lo1 ? lo1 : (il1 > cnt ? cnt : il1);
        const unsigned int jl1 = q1 - il1;
        // load the next tile's first chunks now, so they arrive while this
        // tile is scanned and stored: one more than this tile needed
        {
            const unsigned long long dn = d0 + q1;
            const unsigned int in = i0 + il1;
            loaded = used + 1 < VT ? used + 1 : VT;
            if (dn < d_end) {
                const unsigned int qn = (unsigned int)(d_end - dn < TP ? d_end - dn : TP);
                const unsigned int cn = n - in < qn ? n - in : qn;
#pragma unroll
                for (int m = 0; m < VT; ++m) {
                    if (m >= loaded) break;  // warp-uniform
                    const unsigned int k = (unsigned int)lane + 32u * m;
                    raw[m] = k < cn ? __ldg(ends + in + k) : 0xffffffffu;
                }
            }
        }
        __syncwarp();
        // Inclusive max-scan of the marks over the frame: lane l takes frame
        // positions b0 = VT l .. b0 + VT - 1 (one padded base, VT words on:
        // b0 is a multiple of VT, so the pad is the same for all of them),
        // zeroes its marks as it reads them (every mark lies below the
        // frame's end), and writes its owners straight from registers, two
        // 16-byte stores when all are entries of the tile.
        const unsigned int b0 = (unsigned int)lane * VT;
        unsigned int *mb = buf + pad(b0);
        unsigned int run = 0u, xm[VT];
#pragma unroll
        for (int v = 0; v < VT; ++v) {
            xm[v] = mb[v];
            mb[v] = 0u;
            run = xm[v] > run ? xm[v] : run;
        }
        unsigned int inc = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned int y = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc = y > inc ? y : inc;
        }
        run = __shfl_up_sync(0xffffffffu, inc, 1);
        if (lane == 0) run = 0u;
#pragma unroll
        for (int v = 0; v < VT; ++v) {
            run = xm[v] > run ? xm[v] : run;
            xm[v] = i0 + run;
        }
        // frame position f is owner element j0 + (f - s_al); entries are f in [s_al, s_al + jl1)
        if (b0 >= s_al && b0 + VT <= s_al + jl1) {
            int32_t *dst = owner + j0 + (b0 - s_al);  // 16-byte aligned
#pragma unroll
            for (int v = 0; v < VT; v += 4)
                __stcs(reinterpret_cast<int4 *>(dst + v),
                       make_int4((int)xm[v], (int)xm[v + 1], (int)xm[v + 2], (int)xm[v + 3]));
        } else {
#pragma unroll
            for (int v = 0; v < VT; ++v) {
                const unsigned int f = b0 + v;
                if (f >= s_al && f < s_al + jl1) owner[j0 + (f - s_al)] = (int32_t)xm[v];
            }
        }
        __syncwarp();
        i0 += il1;
        d0 += q1;
    }
}

static std::mutex g_runs_mu;
static int g_runs_sms[64];
static int g_runs_bps[64];

static int runs_grid(int *owner_grid, int *fill_grid) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    std::lock_guard<std::mutex> lock(g_runs_mu);
    if (g_runs_sms[dev] == 0 &&
        cudaDeviceGetAttribute(&g_runs_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return U32SCAN_ECUDA;
    if (g_runs_bps[dev] == 0) {
        int bps = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, runs_owner_kernel<kROWarps, kROVT>, kROThreads,
                                                          0) != cudaSuccess ||
            bps < 1)
            return U32SCAN_ECUDA;
        g_runs_bps[dev] = bps;
    }
    *owner_grid = g_runs_sms[dev] * g_runs_bps[dev];
    *fill_grid = g_runs_sms[dev] * 4;
    return U32SCAN_OK;
}

static bool overlaps(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return a_bytes && b_bytes && x < y + b_bytes && y < x + a_bytes;
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int runs_layout_u32(uint32_t *counts, size_t n, uint32_t *entries, int32_t *slots, size_t slot_capacity,
                               void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    const cudaStream_t s = (cudaStream_t)stream;
    if (n >= (1ull << 31) || entries == nullptr || (n > 0 && counts == nullptr)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(counts) & 3) || (reinterpret_cast<uintptr_t>(entries) & 3) ||
        (reinterpret_cast<uintptr_t>(slots) & 3))
        return U32SCAN_EINVAL;
    const size_t cap = slots ? slot_capacity : 0;
    if (cap >= (1ull << 32)) return U32SCAN_EINVAL;
    if (overlaps(entries, 4, counts, 4 * n) || overlaps(slots, 4 * cap, counts, 4 * n) ||
        overlaps(slots, 4 * cap, entries, 4))
        return U32SCAN_EINVAL;
    int rc = scan_inclusive_launch(counts, n, entries, ws, ws_bytes, s);
    if (rc != U32SCAN_OK) return rc;
    int owner_grid = 0, fill_grid = 0;
    rc = runs_grid(&owner_grid, &fill_grid);
    if (rc != U32SCAN_OK) return rc;
    runs_entries_slots_kernel<<<cap ? fill_grid : 1, kFillThreads, 0, s>>>(entries, cap ? slots : nullptr, cap);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

extern "C" int runs_owner_u32(const uint32_t *ends, size_t n, int32_t *owner, size_t capacity,
                              u32scan_stream_t stream) {
    const cudaStream_t s = (cudaStream_t)stream;
    if (n >= (1ull << 31) || (n > 0 && ends == nullptr) || (capacity > 0 && owner == nullptr)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(ends) & 3) || (reinterpret_cast<uintptr_t>(owner) & 3)) return U32SCAN_EINVAL;
    if (capacity >= (1ull << 32)) return U32SCAN_EINVAL;
    if (overlaps(owner, 4 * capacity, ends, 4 * n)) return U32SCAN_EINVAL;
    if (capacity == 0) return U32SCAN_OK;
    if (n == 0)  // no owners: the one slot of the layout, -1
        return cudaMemsetAsync(owner, 0xff, sizeof(int32_t), s) == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
    int owner_grid = 0, fill_grid = 0;
    const int rc = runs_grid(&owner_grid, &fill_grid);
    if (rc != U32SCAN_OK) return rc;
    runs_owner_kernel<kROWarps, kROVT><<<owner_grid, kROThreads, 0, s>>>(ends, (unsigned int)n, owner, capacity);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

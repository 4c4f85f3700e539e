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
// instead of 32. Per digit pass:
//   upsweep    each 8192-key tile counts its keys per digit value (warp
//              match-any ranking into per-warp counters in shared memory) and
//              writes the 256 counts into a digit-major table;
//   scan       one exclusive scan of that table (the library's own scan
//              kernel) gives every (digit value, tile) its first output slot:
//              all smaller digit values first, then earlier tiles;
//   downsweep  each tile ranks its keys stably within the tile and scatters
//              (key, index) pairs to their slots.
// A histogram of all four digits, taken first, finds digits that are equal
// for every key; their passes are skipped (exact: such a pass moves
// nothing). Which passes run, and which buffers they read and write, is
// decided on the device, so the call stays asynchronous. The last pass
// writes the indices into `perm` and, for radix_sort_u32, the sorted keys
// into `keys_out`; a keys-only sort moves no indices at all.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

constexpr int kRThreads = 512;
constexpr int kRKeys = 16;  // keys per thread per tile
constexpr unsigned int kRTile = kRThreads * kRKeys;
constexpr int kRWarps = kRThreads / 32;

// One pass's role, decided on the device from the histograms.
struct RadixPlan {
    int active;  // this digit differs between keys
    int j;       // index of this pass among the active ones
    int m;       // number of active passes
    int pad;
};

// Workspace layout for n keys (all regions 256-byte aligned). It starts
// with the table scan's own workspace, whose 256-byte header (tile counter,
// call epoch, device status) is the header every operation keeps at offset
// 0, so u32scan_check reads the status of this call and the workspace stays
// valid for any operation afterwards.
struct RadixLayout {
    size_t scan_ws, hist, plan, table, k1, k2, i1, total;
    unsigned int n_tiles;
    explicit RadixLayout(unsigned long long n) {
        n_tiles = (unsigned int)((n + kRTile - 1) / kRTile);
        const unsigned long long cells = 256ull * n_tiles;
        size_t o = 0;
        scan_ws = o;
        o += scan_workspace_bytes(cells);
        hist = o;
        o += round_up(4 * 256 * 4, 256);
        plan = o;
        o += round_up(4 * sizeof(RadixPlan), 256);
        table = o;
        o += round_up(4 * cells, 256);
        k1 = o;
        o += round_up(4 * n, 256);
        k2 = o;
        o += round_up(4 * n, 256);
        i1 = o;
        o += round_up(4 * n, 256);
        total = o;
    }
};

// Counts of all four digits over all keys (one read), for the plan.
__global__ void radix_histogram_kernel(const uint32_t *__restrict__ keys, unsigned long long n,
                                       unsigned int *__restrict__ hist) {
    __shared__ unsigned int s_h[4][256];
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) (&s_h[0][0])[i] = 0;
    __syncthreads();
    auto add = [&](uint32_t k) {
        atomicAdd(&s_h[0][k & 255u], 1u);
        atomicAdd(&s_h[1][(k >> 8) & 255u], 1u);
        atomicAdd(&s_h[2][(k >> 16) & 255u], 1u);
        atomicAdd(&s_h[3][k >> 24], 1u);
    };
    // scalar head up to 16-byte alignment, 16-byte body, scalar tail
    const unsigned long long head = ((16 - (reinterpret_cast<uintptr_t>(keys) & 15)) & 15) / 4;
    const unsigned long long h = head < n ? head : n;
    const unsigned long long nv = (n - h) / 4;
    const unsigned long long gtid = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned long long gstride = (unsigned long long)gridDim.x * blockDim.x;
    if (gtid < h) add(keys[gtid]);
    const uint4 *kv = reinterpret_cast<const uint4 *>(keys + h);
    for (unsigned long long i = gtid; i < nv; i += gstride) {
        const uint4 q = kv[i];
        // a quad whose four keys agree on a digit (common when the digit is
        // constant over the keys) takes one atomic for it instead of four
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const unsigned int s = 8 * p;
            const unsigned int a = (q.x >> s) & 255u, b = (q.y >> s) & 255u, c = (q.z >> s) & 255u,
                               d = (q.w >> s) & 255u;
            if (a == b && b == c && c == d) {
                atomicAdd(&s_h[p][a], 4u);
            } else {
                atomicAdd(&s_h[p][a], 1u);
                atomicAdd(&s_h[p][b], 1u);
                atomicAdd(&s_h[p][c], 1u);
                atomicAdd(&s_h[p][d], 1u);
            }
        }
    }
    for (unsigned long long i = h + 4 * nv + gtid; i < n; i += gstride) add(keys[i]);
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) {
        const unsigned int c = (&s_h[0][0])[i];
        if (c) atomicAdd(hist + i, c);
    }
}

// One warp: a digit is constant when one value holds all n keys.
__global__ void radix_plan_kernel(const unsigned int *__restrict__ hist, unsigned long long n, RadixPlan *plan) {
    const int lane = threadIdx.x & 31;
    int active[4];
    int m = 0;
    for (int p = 0; p < 4; ++p) {
        bool whole = false;
        for (int b = lane; b < 256; b += 32) whole = whole || hist[256 * p + b] == n;
        active[p] = __any_sync(0xffffffffu, whole) ? 0 : 1;
        m += active[p];
    }
    if (lane == 0) {
        int j = 0;
        for (int p = 0; p < 4; ++p) {
            plan[p].active = active[p];
            plan[p].j = j;
            plan[p].m = m;
            j += active[p];
        }
    }
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

// Load this thread's keys of tile t (warp-striped: round r of warp w covers
// 32 consecutive keys) and rank them stably within the tile: after the call
// wrank[r] is the key's rank among the keys of its digit value in this warp
// (in tile order) and s_cnt[w][v] the warp's count of digit value v. Bit r
// of the returned mask says whether key r lies inside the array.
__device__ __forceinline__ unsigned int radix_rank_tile(const uint32_t *__restrict__ in_keys, unsigned long long n,
                                                        unsigned int t, int shift, uint32_t (&k)[kRKeys],
                                                        unsigned int (&wrank)[kRKeys], unsigned int (*s_cnt)[256],
                                                        int lane, int warp) {
    const unsigned long long base = (unsigned long long)t * kRTile + (unsigned long long)warp * (32 * kRKeys);
    for (int i = lane; i < 256; i += 32) s_cnt[warp][i] = 0;
    __syncwarp();
    unsigned int valid_bits = 0;
#pragma unroll
    for (int r = 0; r < kRKeys; ++r) {
        const unsigned long long e = base + 32 * r + lane;
        k[r] = e < n ? in_keys[e] : 0u;
        valid_bits |= (e < n ? 1u : 0u) << r;
    }
#pragma unroll
    for (int r = 0; r < kRKeys; ++r) {
        // lanes holding the same digit value: the AND over the digit's eight
        // bits of the ballot (bit set) or its complement (bit clear), and
        // the same for validity
        const bool valid = (valid_bits >> r) & 1u;
        const unsigned int dr = (k[r] >> shift) & 255u;
        const unsigned int vb = __ballot_sync(0xffffffffu, valid);
        unsigned int same = valid ? vb : ~vb;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const bool bit = (dr >> b) & 1u;
            const unsigned int bb = __ballot_sync(0xffffffffu, bit);
            same &= bit ? bb : ~bb;
        }
        const unsigned int below = (unsigned int)__popc(same & lanemask_lt(lane));
        unsigned int old = 0;
        if (valid) old = s_cnt[warp][dr];
        wrank[r] = old + below;
        __syncwarp();
        if (valid && below == 0) s_cnt[warp][dr] = old + (unsigned int)__popc(same);
        __syncwarp();
    }
    return valid_bits;
}

// Upsweep of one pass: the tile's count of each digit value, written into
// the digit-major table. Counting needs no ranks, so each warp adds its keys
// into its own row of shared-memory counters with atomics.
__global__ void __launch_bounds__(kRThreads, 2)
radix_upsweep_kernel(const RadixPlan *__restrict__ plan, int p, const uint32_t *keys, uint32_t *k1, uint32_t *k2,
                     int32_t *i1, int32_t *perm, uint32_t *keys_out, unsigned long long n, unsigned int n_tiles,
                     unsigned int *__restrict__ table) {
    const RadixPlan pl = plan[p];
    if (!pl.active) return;
    __shared__ unsigned int s_cnt[kRWarps][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const PassBuffers b = pass_buffers(pl, keys, k1, k2, i1, perm, keys_out);
    for (int i = lane; i < 256; i += 32) s_cnt[warp][i] = 0;
    __syncwarp();
    const unsigned long long base = (unsigned long long)blockIdx.x * kRTile + (unsigned long long)warp * (32 * kRKeys);
    uint32_t k[kRKeys];
#pragma unroll
    for (int r = 0; r < kRKeys; ++r) {
        const unsigned long long e = base + 32 * r + lane;
        k[r] = e < n ? b.in_keys[e] : 0u;
    }
    const int shift = 8 * p;
#pragma unroll
    for (int r = 0; r < kRKeys; ++r)
        if (base + 32 * r + lane < n) atomicAdd(&s_cnt[warp][(k[r] >> shift) & 255u], 1u);
    __syncthreads();
    for (int v = threadIdx.x; v < 256; v += kRThreads) {
        unsigned int c = 0;
#pragma unroll
        for (int w = 0; w < kRWarps; ++w) c += s_cnt[w][v];
        table[(unsigned long long)v * n_tiles + blockIdx.x] = c;
    }
}

// Downsweep of one pass: rank the tile, order it by digit value in shared
// memory (stable), then write each digit value's run of (key, index) pairs
// to its slots with consecutive threads on consecutive slots.
__global__ void __launch_bounds__(kRThreads, 2)
radix_downsweep_kernel(const RadixPlan *__restrict__ plan, int p, const uint32_t *keys, uint32_t *k1, uint32_t *k2,
                       int32_t *i1, int32_t *perm, uint32_t *keys_out, unsigned long long n, unsigned int n_tiles,
                       const unsigned int *__restrict__ slots) {
    const RadixPlan pl = plan[p];
    if (!pl.active) return;
    extern __shared__ __align__(16) unsigned int r_smem[];
    unsigned int(*s_cnt)[256] = reinterpret_cast<unsigned int(*)[256]>(r_smem);  // [kRWarps][256]
    unsigned int *s_tileoff = r_smem + kRWarps * 256;                           // [256] digit start in tile
    unsigned int *s_glob = s_tileoff + 256;                                     // [256] digit's first slot
    unsigned int *s_keys = s_glob + 256;                                        // [kRTile]
    int32_t *s_idx = reinterpret_cast<int32_t *>(s_keys + kRTile);              // [kRTile]
    __shared__ unsigned int s_part[kRThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned int t = blockIdx.x;
    const PassBuffers b = pass_buffers(pl, keys, k1, k2, i1, perm, keys_out);
    uint32_t k[kRKeys];
    unsigned int wrank[kRKeys];
    const unsigned int valid_bits = radix_rank_tile(b.in_keys, n, t, 8 * p, k, wrank, s_cnt, lane, warp);
    __syncthreads();
    // Per digit value v (threads 0..255): warp offsets within the value's
    // run in this tile, and the run's length; then the runs' starts.
    unsigned int tot = 0;
    if (threadIdx.x < 256) {
        const int v = threadIdx.x;
#pragma unroll
        for (int w = 0; w < kRWarps; ++w) {
            const unsigned int c = s_cnt[w][v];
            s_cnt[w][v] = tot;
            tot += c;
        }
        s_glob[v] = slots[(unsigned long long)v * n_tiles + t];
    }
    // exclusive scan of the 256 run lengths over threads 0..255
    const unsigned int inc = warp_inclusive_sum(tot, lane);
    if (lane == 31 && threadIdx.x < 256) s_part[warp] = inc;
    __syncthreads();
    if (threadIdx.x < 256) {
        unsigned int before = 0;
        for (int w = 0; w < warp; ++w) before += s_part[w];
        s_tileoff[threadIdx.x] = before + inc - tot;
    }
    __syncthreads();
    const unsigned long long base = (unsigned long long)t * kRTile + (unsigned long long)warp * (32 * kRKeys);
#pragma unroll
    for (int r = 0; r < kRKeys; ++r) {
        if ((valid_bits >> r) & 1u) {
            const unsigned long long e = base + 32 * r + lane;
            const unsigned int v = (k[r] >> (8 * p)) & 255u;
            const unsigned int pos = s_tileoff[v] + s_cnt[warp][v] + wrank[r];
            s_keys[pos] = k[r];
            if (b.out_idx) s_idx[pos] = b.in_idx ? b.in_idx[e] : (int32_t)e;
        }
    }
    __syncthreads();
    const unsigned long long tile0 = (unsigned long long)t * kRTile;
    const unsigned int count = n - tile0 < kRTile ? (unsigned int)(n - tile0) : kRTile;
    const int shift = 8 * p;
    for (unsigned int i = threadIdx.x; i < count; i += kRThreads) {
        const unsigned int key = s_keys[i];
        const unsigned int v = (key >> shift) & 255u;
        const unsigned int slot = s_glob[v] + (i - s_tileoff[v]);
        if (b.out_keys) b.out_keys[slot] = key;
        if (b.out_idx) b.out_idx[slot] = s_idx[i];
    }
}

constexpr size_t kRDownSmem = (size_t)(kRWarps * 256 + 512 + 2 * kRTile) * 4;

// All digits constant (every key equal): the permutation is the identity.
__global__ void radix_identity_kernel(const RadixPlan *__restrict__ plan, const uint32_t *keys, int32_t *perm,
                                      uint32_t *keys_out, unsigned long long n) {
    if (plan[0].m != 0) return;
    for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (unsigned long long)gridDim.x * blockDim.x) {
        if (perm) perm[i] = (int32_t)i;
        if (keys_out) keys_out[i] = keys[i];
    }
}

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
    unsigned int *hist = reinterpret_cast<unsigned int *>(w + L.hist);
    RadixPlan *plan = reinterpret_cast<RadixPlan *>(w + L.plan);
    unsigned int *table = reinterpret_cast<unsigned int *>(w + L.table);
    uint32_t *k1 = reinterpret_cast<uint32_t *>(w + L.k1);
    uint32_t *k2 = reinterpret_cast<uint32_t *>(w + L.k2);
    int32_t *i1 = reinterpret_cast<int32_t *>(w + L.i1);
    {
        static std::mutex mu;
        static bool attr_set[64];
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(radix_downsweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kRDownSmem) != cudaSuccess)
                return U32SCAN_ECUDA;
            attr_set[dev] = true;
        }
    }
    if (cudaMemsetAsync(hist, 0, 4 * 256 * 4, stream) != cudaSuccess) return U32SCAN_ECUDA;
    radix_histogram_kernel<<<1024, 512, 0, stream>>>(keys, n, hist);
    radix_plan_kernel<<<1, 32, 0, stream>>>(hist, n, plan);
    const unsigned long long cells = 256ull * L.n_tiles;
    for (int p = 0; p < 4; ++p) {
        radix_upsweep_kernel<<<L.n_tiles, kRThreads, 0, stream>>>(plan, p, keys, k1, k2, i1, perm, keys_out, n,
                                                                   L.n_tiles, table);
        const int rc = scan_exclusive_launch(table, cells, w + L.scan_ws, scan_workspace_bytes(cells), stream);
        if (rc != U32SCAN_OK) return rc;
        radix_downsweep_kernel<<<L.n_tiles, kRThreads, kRDownSmem, stream>>>(plan, p, keys, k1, k2, i1, perm,
                                                                              keys_out, n, L.n_tiles, table);
    }
    radix_identity_kernel<<<1024, 256, 0, stream>>>(plan, keys, perm, keys_out, n);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
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

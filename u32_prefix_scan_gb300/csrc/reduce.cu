// reduce.cu -- the fold of a U32 array under one of the CAIRN integer
// operators, reading each element once.
//
// Source: the CAIRN "Concurrency" page, section "reduce and compact":
// `reduce` folds a row with add_wrap, mul_wrap, &, |, ^, min or max (sums
// and products wrap at 2^32). Each is associative and commutative, so the
// fold may be taken in any grouping and order and gives the same bits.
//
// count_nonzero_u32 folds (x != 0) with add instead: the number of kept
// elements of a compaction (the entelechy `compact` graph's count), read
// without writing offsets.
//
// Kernel: a grid of resident blocks strides over the array with four 16-byte
// loads in flight a thread; each block folds its share (lanes, then warps)
// into one partial in the workspace, and the last block to finish (counted
// in the workspace header) folds the partials into the total and zeroes
// them. 4 bytes read per element; nothing else but the partials moves.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

constexpr int kFThreads = 512;
constexpr int kFMaxGrid = 1024;  // partials in the workspace

size_t reduce_workspace_bytes() { return kHeaderBytes + round_up(4 * kFMaxGrid, 256); }

// NZ: fold (x != 0) instead of x (with OP = add: the count of non-zero
// elements, the kept count of a compaction).
template <int OP, bool NZ>
__global__ void __launch_bounds__(kFThreads, 2)
reduce_u32_kernel(const uint32_t *__restrict__ data, unsigned long long n, uint32_t *total, WsHeader *hdr,
                  unsigned int *partials) {
    using M = Monoid<OP>;
    __shared__ unsigned int s_warp[kFThreads / 32];
    __shared__ unsigned int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // scalar head up to 16-byte alignment, 16-byte body, scalar tail
    const unsigned long long head = ((16 - (reinterpret_cast<uintptr_t>(data) & 15)) & 15) / 4;
    const unsigned long long h = head < n ? head : n;
    const unsigned long long nv = (n - h) / 4;
    const unsigned long long gtid = (unsigned long long)blockIdx.x * kFThreads + threadIdx.x;
    const unsigned long long gstride = (unsigned long long)gridDim.x * kFThreads;
    auto val = [](unsigned int x) -> unsigned int { return NZ ? (x != 0u ? 1u : 0u) : x; };
    unsigned int acc = M::identity();
    if (gtid < h) acc = M::apply(acc, val(data[gtid]));
    const uint4 *dv = reinterpret_cast<const uint4 *>(data + h);
    auto fold4 = [&](const uint4 &q) {
        acc = M::apply(acc, M::apply(M::apply(val(q.x), val(q.y)), M::apply(val(q.z), val(q.w))));
    };
    unsigned long long i = gtid;
    for (; i + 3 * gstride < nv; i += 4 * gstride) {
        const uint4 q0 = __ldcs(dv + i), q1 = __ldcs(dv + i + gstride), q2 = __ldcs(dv + i + 2 * gstride),
                    q3 = __ldcs(dv + i + 3 * gstride);
        fold4(q0);
        fold4(q1);
        fold4(q2);
        fold4(q3);
    }
    for (; i < nv; i += gstride) fold4(__ldcs(dv + i));
    for (unsigned long long j = h + 4 * nv + gtid; j < n; j += gstride) acc = M::apply(acc, val(data[j]));
    acc = M::warp_fold(acc);
    if (lane == 0) s_warp[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int b = M::identity();
        for (int w = 0; w < kFThreads / 32; ++w) b = M::apply(b, s_warp[w]);
        st_relaxed_u32(partials + blockIdx.x, b);
        __threadfence();
        const bool last = atom_add_acq_rel(&hdr->done, 1u) == gridDim.x - 1u;
        if (last) st_relaxed_u32(&hdr->done, 0u);
        s_last = last ? 1u : 0u;
    }
    __syncthreads();
    if (s_last == 0u) return;
    // the last block folds every block's partial and zeroes it: the partials
    // lie where other operations keep tagged tile words, and two of them
    // side by side could pass for such a word of a later launch
    unsigned int f = M::identity();
    for (unsigned int k = threadIdx.x; k < gridDim.x; k += kFThreads) {
        f = M::apply(f, ld_relaxed_u32(partials + k));
        st_relaxed_u32(partials + k, 0u);
    }
    f = M::warp_fold(f);
    if (lane == 0) s_warp[warp] = f;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int b = M::identity();
        for (int w = 0; w < kFThreads / 32; ++w) b = M::apply(b, s_warp[w]);
        *total = b;
    }
}

static std::mutex g_red_mu;
static int g_red_grid[64];

template <int OP, bool NZ = false>
static int reduce_launch(const uint32_t *data, unsigned long long n, uint32_t *total, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
    if ((n > 0 && data == nullptr) || total == nullptr || n >= (1ull << 62)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(data) & 3) || (reinterpret_cast<uintptr_t>(total) & 3)) return U32SCAN_EINVAL;
    if (n == 0) {  // the fold of nothing is the operator's identity
        const unsigned int id = OP == kMul ? 1u : (OP == kAnd || OP == kMin) ? 0xffffffffu : 0u;
        if (cudaMemsetAsync(total, id == 0xffffffffu ? 0xff : 0, sizeof(uint32_t), stream) != cudaSuccess)
            return U32SCAN_ECUDA;
        if (id == 1u) {
            // one byte of 1 in the low byte (little-endian) makes the word 1
            if (cudaMemsetAsync(total, 1, 1, stream) != cudaSuccess) return U32SCAN_ECUDA;
        }
        return U32SCAN_OK;
    }
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < reduce_workspace_bytes())
        return U32SCAN_EWORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    int grid;
    {
        std::lock_guard<std::mutex> lock(g_red_mu);
        if (g_red_grid[dev] == 0) {
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return U32SCAN_ECUDA;
            g_red_grid[dev] = 2 * sms < kFMaxGrid ? 2 * sms : kFMaxGrid;
        }
        grid = g_red_grid[dev];
    }
    // no more blocks than 16-byte loads (4 a thread), at least one
    const unsigned long long want = (n / 4 + 4ull * kFThreads - 1) / (4ull * kFThreads);
    if (want < (unsigned long long)grid) grid = want > 0 ? (int)want : 1;
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    unsigned int *partials = reinterpret_cast<unsigned int *>(static_cast<char *>(ws) + kHeaderBytes);
    reduce_u32_kernel<OP, NZ><<<grid, kFThreads, 0, stream>>>(data, n, total, hdr, partials);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int reduce_u32_op(int op, const uint32_t *data, size_t n, uint32_t *total, void *ws, size_t ws_bytes,
                             u32scan_stream_t stream) {
    const cudaStream_t s = (cudaStream_t)stream;
    switch (op) {
    case kAdd: return reduce_launch<kAdd>(data, n, total, ws, ws_bytes, s);
    case kMul: return reduce_launch<kMul>(data, n, total, ws, ws_bytes, s);
    case kAnd: return reduce_launch<kAnd>(data, n, total, ws, ws_bytes, s);
    case kOr: return reduce_launch<kOr>(data, n, total, ws, ws_bytes, s);
    case kXor: return reduce_launch<kXor>(data, n, total, ws, ws_bytes, s);
    case kMin: return reduce_launch<kMin>(data, n, total, ws, ws_bytes, s);
    case kMax: return reduce_launch<kMax>(data, n, total, ws, ws_bytes, s);
    default: return U32SCAN_EINVAL;
    }
}

extern "C" int count_nonzero_u32(const uint32_t *data, size_t n, uint32_t *count, void *ws, size_t ws_bytes,
                                 u32scan_stream_t stream) {
    return reduce_launch<kAdd, true>(data, n, count, ws, ws_bytes, (cudaStream_t)stream);
}

// segshard.cu -- the pieces of a segmented scan split across ranks.
//
// Source: "Futhark.Pass.ExtractKernels.Segmented" (regularSegmentedScan)
// for the operation, and the scan.bend source's Driver (block sums, a scan
// of the sums, each block finished from its base) for the composition one
// level up. A piece of a longer array is first scanned on its own with
// segscan_inclusive_u32 (its element 0 opening a segment). What the piece
// passes on is the segmented operator's value over it: whether it holds a
// head, and its last element's scanned value. The segmented exclusive scan
// of the pieces' values gives each piece its carry-in, the segmented value
// flowing into its element 0; only the elements before the piece's first
// head depend on it, and the fix adds it to them:
//
//   piece r holds a head:  carry(r + 1) = tail(r)
//   otherwise:             carry(r + 1) = carry(r) + tail(r)
//
// so the pieces put back together hold the scan of the whole array.
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

// One thread: the piece's summary (has-head, tail, segment count).
__global__ void segshard_summary_kernel(const uint32_t *scanned, const int32_t *flags, unsigned long long n,
                                        const uint32_t *nseg, int first_opens, uint32_t *summary) {
    if (n == 0) {
        summary[0] = 0u;
        summary[1] = 0u;
        summary[2] = 0u;
        return;
    }
    const unsigned int local = *nseg;  // counts element 0 as a head
    const bool head0 = flags[0] != 0;
    summary[0] = (local > 1u || head0) ? 1u : 0u;
    summary[1] = scanned[n - 1];
    summary[2] = (first_opens || head0) ? local : local - 1u;
}

// One thread: the pieces' carries, in order, and the whole segment count.
__global__ void segshard_carries_kernel(const uint32_t *summaries, unsigned long long g, uint32_t *carries,
                                        uint32_t *nseg_total) {
    unsigned int c = 0u, total = 0u;
    for (unsigned long long r = 0; r < g; ++r) {
        carries[r] = c;
        const uint32_t *s = summaries + 3 * r;
        c = s[0] ? s[1] : c + s[1];
        total += s[2];
    }
    if (nseg_total) *nseg_total = total;
}

// The first head of the piece: blocks take 8192-flag chunks in order and
// stop once a head was found before their chunk. Two spare header words
// (bytes 20..27, which no other kernel uses) hold the first head found so
// far (n when none) and the chunk counter, set before the launch.
constexpr unsigned int kFixChunk = 8192;
constexpr int kFixThreads = 512;

__device__ __forceinline__ unsigned int *fix_words(WsHeader *hdr) {
    return reinterpret_cast<unsigned int *>(hdr) + 5;
}
static_assert(offsetof(WsHeader, done) == 16 && offsetof(WsHeader, seg_count) >= 28,
              "bytes 20..27 of the header are spare");

__global__ void fix_init_kernel(WsHeader *hdr, unsigned int n) {
    fix_words(hdr)[0] = n;
    fix_words(hdr)[1] = 0u;
}

__global__ void __launch_bounds__(kFixThreads)
segshard_first_head_kernel(const int32_t *flags, unsigned long long n, WsHeader *hdr) {
    __shared__ unsigned int s_chunk, s_first, s_stop;
    unsigned int *first = fix_words(hdr), *counter = fix_words(hdr) + 1;
    const unsigned long long n_chunks = (n + kFixChunk - 1) / kFixChunk;
    for (;;) {
        if (threadIdx.x == 0) {
            const unsigned int c = atomicAdd(counter, 1u);
            s_chunk = c;
            s_first = 0xffffffffu;
            // past the end, or a head already found before this chunk: stop
            s_stop = ((unsigned long long)c >= n_chunks ||
                      (unsigned long long)ld_relaxed_u32(first) < (unsigned long long)c * kFixChunk)
                         ? 1u
                         : 0u;
        }
        __syncthreads();
        if (s_stop) break;  // the same for every thread of the block
        const unsigned long long c0 = (unsigned long long)s_chunk * kFixChunk;
        const unsigned long long c1 = c0 + kFixChunk < n ? c0 + kFixChunk : n;
        unsigned int mine = 0xffffffffu;
        for (unsigned long long i = c0 + threadIdx.x; i < c1; i += kFixThreads)
            if (flags[i] != 0) {
                mine = (unsigned int)(i - c0);
                break;
            }
        atomicMin(&s_first, mine);
        __syncthreads();
        if (threadIdx.x == 0 && s_first != 0xffffffffu) atomicMin(first, (unsigned int)(c0 + s_first));
        __syncthreads();
    }
}

// Adds the carry to every element before the first head.
__global__ void segshard_add_kernel(uint32_t *data, WsHeader *hdr, const uint32_t *carry) {
    const unsigned long long first = ld_relaxed_u32(fix_words(hdr));
    const unsigned int c = *carry;
    if (c == 0u) return;
    for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < first;
         i += (unsigned long long)gridDim.x * blockDim.x)
        data[i] += c;
}

static std::mutex g_fix_mu;
static int g_fix_sms[64];

}  // namespace u32scan

using namespace u32scan;

extern "C" int segscan_piece_summary_u32(const uint32_t *scanned, const int32_t *head_flags, size_t n,
                                         const uint32_t *nseg, int first_opens, uint32_t *summary,
                                         u32scan_stream_t stream) {
    if (summary == nullptr || (n > 0 && (scanned == nullptr || head_flags == nullptr || nseg == nullptr)))
        return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(scanned) & 3) || (reinterpret_cast<uintptr_t>(head_flags) & 3) ||
        (reinterpret_cast<uintptr_t>(nseg) & 3) || (reinterpret_cast<uintptr_t>(summary) & 3))
        return U32SCAN_EINVAL;
    segshard_summary_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(scanned, head_flags, n, nseg, first_opens,
                                                               summary);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

extern "C" int segscan_piece_carries_u32(const uint32_t *summaries, size_t g, uint32_t *carries,
                                         uint32_t *nseg_total, u32scan_stream_t stream) {
    if (g > 0 && (summaries == nullptr || carries == nullptr)) return U32SCAN_EINVAL;
    if (g == 0 && nseg_total == nullptr) return U32SCAN_OK;
    if ((reinterpret_cast<uintptr_t>(summaries) & 3) || (reinterpret_cast<uintptr_t>(carries) & 3) ||
        (reinterpret_cast<uintptr_t>(nseg_total) & 3))
        return U32SCAN_EINVAL;
    segshard_carries_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(summaries, g, carries, nseg_total);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

extern "C" int segscan_fix_u32(uint32_t *data, const int32_t *head_flags, size_t n, const uint32_t *carry,
                               void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    const cudaStream_t s = (cudaStream_t)stream;
    if (n >= (1ull << 32) || (n > 0 && (data == nullptr || head_flags == nullptr || carry == nullptr)))
        return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(data) & 3) || (reinterpret_cast<uintptr_t>(head_flags) & 3) ||
        (reinterpret_cast<uintptr_t>(carry) & 3))
        return U32SCAN_EINVAL;
    if (n == 0) return U32SCAN_OK;
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < kHeaderBytes)
        return U32SCAN_EWORKSPACE;
    int dev = -1, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    {
        std::lock_guard<std::mutex> lock(g_fix_mu);
        if (g_fix_sms[dev] == 0 &&
            cudaDeviceGetAttribute(&g_fix_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return U32SCAN_ECUDA;
        sms = g_fix_sms[dev];
    }
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    fix_init_kernel<<<1, 1, 0, s>>>(hdr, (unsigned int)n);
    const unsigned long long chunks = (n + kFixChunk - 1) / kFixChunk;
    const unsigned int grid = chunks < (unsigned long long)(2 * sms) ? (unsigned int)chunks : (unsigned int)(2 * sms);
    segshard_first_head_kernel<<<grid, kFixThreads, 0, s>>>(head_flags, n, hdr);
    segshard_add_kernel<<<2 * sms, 256, 0, s>>>(data, hdr, carry);
    // leave the spare words zero, as a zero-filled header has them
    if (cudaMemsetAsync(reinterpret_cast<unsigned int *>(hdr) + 5, 0, 2 * sizeof(unsigned int), s) != cudaSuccess)
        return U32SCAN_ECUDA;
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

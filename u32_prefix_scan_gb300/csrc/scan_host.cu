// scan_host.cu -- exclusive and inclusive U32 scans of arrays in host memory.
//
// Source: "scan.bend source" (bendlib), section API (`exclusive`,
// `inclusive`, the total) and the header comment (sums wrap at 2^32), as for
// the device-resident scans; the pages keep their arrays in device memory,
// and this file only moves a host array through the device scan.
//
// On GB300 the host link (NVLink-C2C to the Grace CPU) moves about 170-210
// GB/s per direction, some thirty times less than HBM, so a host-to-host scan
// is bound by the two copies. The array is cut into chunks that flow
// through a ring of device staging slots in the caller's workspace, on three
// streams ordered by events:
//
//   copy-in stream   H2D chunk j into slot j % R (after chunk j - R left it)
//   caller's stream  scan chunk j in its slot, after the carry of chunk j - 1
//   copy-out stream  D2H chunk j from its slot
//
// so the copy in of chunk j + 1, the scan of chunk j and the copy out of
// chunk j - 1 overlap. Chunk j's scan folds in the wrapped sum of all earlier
// chunks (a device carry word written by chunk j - 1's scan), so the chunks
// chain into one scan of the whole array with one read and one write of each
// element on each side of the link.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

// Chunk sizes in elements: at most 2^23 (32 MiB, about 0.2 ms on the link
// each way), at least 2^18, else about an eighth of the array so that short
// arrays still overlap their copies. Each chunk costs about 6.5 us beyond
// its bytes (measured on GB300 at n = 2^28: 2^20-element chunks 8.0 ms,
// 2^21 7.4, 2^22 6.96, 2^23 6.75), so chunks are as long as the fill and
// drain of the pipeline allow. Staging slots: one being copied in, one
// being scanned, one being copied out, and a spare (3, 4 and 8 slots
// measured alike). Both can be overridden at build time for sweeps.
#ifndef U32SCAN_H_CHUNK_LOG2
#define U32SCAN_H_CHUNK_LOG2 23
#endif
#ifndef U32SCAN_H_RING
#define U32SCAN_H_RING 4
#endif
constexpr unsigned long long kHostChunkMax = 1ull << U32SCAN_H_CHUNK_LOG2;
constexpr unsigned long long kHostChunkMin = 1ull << 18;
constexpr unsigned long long kHostRing = U32SCAN_H_RING;
static_assert(U32SCAN_H_CHUNK_LOG2 >= 18 && kHostRing >= 1, "chunks of at least 2^18 elements");

static unsigned long long host_chunk(unsigned long long n) {
    unsigned long long c = round_up((n + 7) / 8, 64);
    if (c < kHostChunkMin) c = kHostChunkMin;
    if (c > kHostChunkMax) c = kHostChunkMax;
    if (c > n) c = round_up(n, 64);
    return c;
}

struct HostLayout {
    unsigned long long chunk, chunks, slots;
    size_t scan_ws, chain_off, ring_off, bytes;
};

static HostLayout host_layout(unsigned long long n) {
    HostLayout L{};
    L.chunk = host_chunk(n);
    L.chunks = L.chunk ? (n + L.chunk - 1) / L.chunk : 0;
    L.slots = L.chunks < kHostRing ? L.chunks : kHostRing;
    L.scan_ws = round_up(scan_workspace_bytes_upto(L.chunk ? L.chunk : 1), 256);
    L.chain_off = L.scan_ws;           // two carry words, ping-pong between chunks
    L.ring_off = L.chain_off + 256;    // staging slots, 256-byte aligned
    L.bytes = L.ring_off + L.slots * L.chunk * 4;
    return L;
}

size_t scan_host_workspace_bytes(unsigned long long n) { return host_layout(n).bytes; }

// True when [p, p + bytes) lies in page-locked host memory known to CUDA
// (cudaHostAlloc, cudaMallocHost, cudaHostRegister): both ends are checked.
static bool page_locked(const void *p, size_t bytes) {
    const char *c = static_cast<const char *>(p);
    const void *ends[2] = {c, c + bytes - 1};
    for (const void *e : ends) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, e) != cudaSuccess) {
            (void)cudaGetLastError();  // clear the query's (non-sticky) error
            return false;
        }
        if (a.type != cudaMemoryTypeHost) return false;
    }
    return true;
}

static bool overlap(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

// Streams and events of one call. They are created per call and destroyed
// at its end; CUDA releases each one once the work queued on it completes,
// so the call stays asynchronous.
struct Pipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done_in = nullptr, done_out = nullptr;
    cudaEvent_t loaded[kHostRing] = {}, scanned[kHostRing] = {}, stored[kHostRing] = {};

    bool create() {
        const unsigned f = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) != cudaSuccess) return false;
        if (cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(&start, f) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(&done_in, f) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(&done_out, f) != cudaSuccess) return false;
        for (unsigned long long i = 0; i < kHostRing; ++i)
            if (cudaEventCreateWithFlags(&loaded[i], f) != cudaSuccess ||
                cudaEventCreateWithFlags(&scanned[i], f) != cudaSuccess ||
                cudaEventCreateWithFlags(&stored[i], f) != cudaSuccess)
                return false;
        return true;
    }
    // Order everything later on `s` after all work queued on the two copy
    // streams, then release the handles.
    bool join(cudaStream_t s) {
        bool ok = true;
        if (in && done_in) ok &= cudaEventRecord(done_in, in) == cudaSuccess && cudaStreamWaitEvent(s, done_in, 0) == cudaSuccess;
        if (out && done_out) ok &= cudaEventRecord(done_out, out) == cudaSuccess && cudaStreamWaitEvent(s, done_out, 0) == cudaSuccess;
        return ok;
    }
    ~Pipe() {
        for (unsigned long long i = 0; i < kHostRing; ++i) {
            if (loaded[i]) cudaEventDestroy(loaded[i]);
            if (scanned[i]) cudaEventDestroy(scanned[i]);
            if (stored[i]) cudaEventDestroy(stored[i]);
        }
        if (start) cudaEventDestroy(start);
        if (done_in) cudaEventDestroy(done_in);
        if (done_out) cudaEventDestroy(done_out);
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
    }
};

static void CUDART_CB zero_word(void *p) { *static_cast<uint32_t *>(p) = 0u; }

static int scan_host(bool inclusive, const uint32_t *host_in, uint32_t *host_out, size_t n, uint32_t *host_total,
                     void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (n > 0 && (host_in == nullptr || host_out == nullptr)) return U32SCAN_EINVAL;
    if (n >= (1ull << 62)) return U32SCAN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(host_in) & 3) || (reinterpret_cast<uintptr_t>(host_out) & 3) ||
        (reinterpret_cast<uintptr_t>(host_total) & 3))
        return U32SCAN_EINVAL;
    const size_t bytes = 4 * n;
    if (n > 0) {
        if (host_in != host_out && overlap(host_in, bytes, host_out, bytes)) return U32SCAN_EINVAL;
        if (!page_locked(host_in, bytes) || !page_locked(host_out, bytes)) return U32SCAN_EINVAL;
    }
    if (host_total) {
        if (!page_locked(host_total, 4)) return U32SCAN_EINVAL;
        if (n > 0 && (overlap(host_total, 4, host_in, bytes) || overlap(host_total, 4, host_out, bytes)))
            return U32SCAN_EINVAL;
    }
    if (n == 0) {  // total 0, written in stream order; nothing else to do
        if (host_total && cudaLaunchHostFunc(stream, zero_word, host_total) != cudaSuccess) return U32SCAN_ECUDA;
        return U32SCAN_OK;
    }
    const HostLayout L = host_layout(n);
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < L.bytes) return U32SCAN_EWORKSPACE;
    char *w = static_cast<char *>(ws);
    uint32_t *chain = reinterpret_cast<uint32_t *>(w + L.chain_off);
    uint32_t *ring = reinterpret_cast<uint32_t *>(w + L.ring_off);

    Pipe P;
    if (!P.create()) return U32SCAN_ECUDA;
    // Both copy streams start after the work already queued on `stream`.
    bool ok = cudaEventRecord(P.start, stream) == cudaSuccess && cudaStreamWaitEvent(P.in, P.start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(P.out, P.start, 0) == cudaSuccess;
    int rc = U32SCAN_OK;
    for (unsigned long long j = 0; ok && j < L.chunks; ++j) {
        const unsigned long long k = j % L.slots;
        const unsigned long long off = j * L.chunk;
        const unsigned long long len = n - off < L.chunk ? n - off : L.chunk;
        uint32_t *slot = ring + k * L.chunk;
        // Copy in, once the slot's previous chunk has been copied out.
        if (j >= L.slots) ok = ok && cudaStreamWaitEvent(P.in, P.stored[k], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(slot, host_in + off, 4 * len, cudaMemcpyHostToDevice, P.in) == cudaSuccess;
        ok = ok && cudaEventRecord(P.loaded[k], P.in) == cudaSuccess;
        // Scan on the caller's stream, after the carry of the chunks before.
        ok = ok && cudaStreamWaitEvent(stream, P.loaded[k], 0) == cudaSuccess;
        if (ok) {
            rc = scan_chunk_launch(inclusive, slot, len, j == 0 ? nullptr : chain + ((j - 1) & 1), chain + (j & 1),
                                   ws, L.scan_ws, stream);
            ok = rc == U32SCAN_OK;
        }
        ok = ok && cudaEventRecord(P.scanned[k], stream) == cudaSuccess;
        // Copy out.
        ok = ok && cudaStreamWaitEvent(P.out, P.scanned[k], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(host_out + off, slot, 4 * len, cudaMemcpyDeviceToHost, P.out) == cudaSuccess;
        ok = ok && cudaEventRecord(P.stored[k], P.out) == cudaSuccess;
    }
    if (ok && host_total)  // the last chunk's total is the array's
        ok = cudaMemcpyAsync(host_total, chain + ((L.chunks - 1) & 1), 4, cudaMemcpyDeviceToHost, P.out) == cudaSuccess;
    // Whatever was queued, later work on `stream` comes after it.
    const bool joined = P.join(stream);
    if (rc != U32SCAN_OK) return rc;
    if (!ok || !joined) return U32SCAN_ECUDA;
    // The carry words and the staging slots hold plain data (the scanned
    // chunks) where other operations keep tagged tile words; two values side
    // by side could pass for such a word. Zero that part once the copies out
    // are done (the slots past it no operation reads as tile words).
    const size_t reach = tile_word_reach();
    const size_t end = L.bytes < reach ? L.bytes : reach;
    if (end > L.chain_off && cudaMemsetAsync(w + L.chain_off, 0, end - L.chain_off, stream) != cudaSuccess)
        return U32SCAN_ECUDA;
    return U32SCAN_OK;
}

}  // namespace u32scan

using namespace u32scan;

extern "C" int scan_exclusive_u32_host(const uint32_t *host_in, uint32_t *host_out, size_t n, uint32_t *host_total,
                                       void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    return scan_host(false, host_in, host_out, n, host_total, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int scan_inclusive_u32_host(const uint32_t *host_in, uint32_t *host_out, size_t n, uint32_t *host_total,
                                       void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    return scan_host(true, host_in, host_out, n, host_total, ws, ws_bytes, (cudaStream_t)stream);
}

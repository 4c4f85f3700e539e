// api.cu -- the library-wide entry points: workspace sizing and set-up,
// device-status readout, error strings, version.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

// The largest span, from the workspace start, that any operation's tile
// words can take: the largest workspace of the operations that keep nothing
// but tile words there, over every n below 2^32 (a few MiB).
size_t tile_word_reach() {
    size_t reach = scan_workspace_bytes(0xffffffffull);
    for (const size_t b : {segscan_workspace_bytes(0xffffffffull), compact_workspace_bytes(0xffffffffull),
                           compact_values_workspace_bytes(0xffffffffull), scan64_workspace_bytes(0xffffffffull)})
        reach = b > reach ? b : reach;
    return reach;
}

unsigned long long tile_words_to_clear(size_t ws_bytes) {
    const size_t reach = tile_word_reach();
    const size_t end = ws_bytes < reach ? ws_bytes : reach;
    return end > kHeaderBytes ? (end - kHeaderBytes) / 8 : 0ull;
}

}  // namespace u32scan

using namespace u32scan;

extern "C" size_t u32scan_workspace_bytes(int op, size_t n) {
    switch (op) {
    case U32SCAN_OP_SCAN:
        return scan_workspace_bytes(n);
    case U32SCAN_OP_SEGSCAN:
        return segscan_workspace_bytes(n);
    case U32SCAN_OP_COMPACT: {
        const size_t a = compact_workspace_bytes(n), b = compact_values_workspace_bytes(n);
        return a > b ? a : b;
    }
    case U32SCAN_OP_RADIX:
        return radix_workspace_bytes(n);
    case U32SCAN_OP_RUNS:
        return scan_workspace_bytes(n);
    case U32SCAN_OP_SCAN64:
        return scan64_workspace_bytes(n);
    case U32SCAN_OP_SCAN_HOST:
        return scan_host_workspace_bytes(n);
    case U32SCAN_OP_REDUCE:
        return reduce_workspace_bytes();
    default:
        return 0;
    }
}

extern "C" int u32scan_workspace_init(void *ws, size_t ws_bytes, u32scan_stream_t stream) {
    if (ws == nullptr || ws_bytes < kHeaderBytes) return U32SCAN_EWORKSPACE;
    return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

extern "C" int u32scan_check(void *ws, u32scan_stream_t stream) {
    if (ws == nullptr) return U32SCAN_EWORKSPACE;
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    unsigned int status = 0;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return U32SCAN_ECUDA;
    if (cudaMemcpy(&status, &hdr->status, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
        return U32SCAN_ECUDA;
    if (status == 0) return U32SCAN_OK;
    const unsigned int zero[2] = {0u, 0u};
    if (cudaMemcpy(&hdr->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return U32SCAN_ECUDA;
    return (status & kStatusTimeout) ? U32SCAN_ETIMEOUT : U32SCAN_ECUDA;
}

extern "C" const char *u32scan_strerror(int status) {
    switch (status) {
    case U32SCAN_OK:
        return "ok";
    case U32SCAN_EINVAL:
        return "invalid argument (null pointer, misaligned pointer or n out of range)";
    case U32SCAN_EWORKSPACE:
        return "workspace missing, misaligned or smaller than u32scan_workspace_bytes";
    case U32SCAN_ECUDA:
        return "CUDA runtime error";
    case U32SCAN_ETIMEOUT:
        return "a wait timed out (a predecessor's carry or a tile's bulk copy): the results of the calls "
               "since the last check are invalid; zero-fill the workspace before reusing it";
    default:
        return "unknown status";
    }
}

extern "C" int u32scan_version(void) { return 100; }

/*
 * scan_in_place.c -- calling libu32scan from C.
 *
 * An in-place exclusive scan of n device words: size and zero-fill a
 * workspace once, make the call, read the device-side status. Build with
 *   cc -std=c99 scan_in_place.c -I include -I /usr/local/cuda/include \
 *      u32_prefix_scan_gb300/libu32scan.so -L /usr/local/cuda/lib64 -lcudart
 */
#include <cuda_runtime.h>
#include "u32scan.h"

/* In-place exclusive scan of n device words; the total lands in *d_total. */
int scan_in_place(uint32_t *d_data, size_t n, uint32_t *d_total, cudaStream_t s)
{
    size_t ws_bytes = u32scan_workspace_bytes(U32SCAN_OP_SCAN, n);
    void *ws = NULL;
    if (cudaMalloc(&ws, ws_bytes) != cudaSuccess) return U32SCAN_ECUDA;
    int rc = u32scan_workspace_init(ws, ws_bytes, (u32scan_stream_t)s);  /* once per workspace */
    if (rc == U32SCAN_OK) rc = scan_exclusive_u32(d_data, n, d_total, ws, ws_bytes, (u32scan_stream_t)s);
    if (rc == U32SCAN_OK) rc = u32scan_check(ws, (u32scan_stream_t)s);   /* syncs s; device status */
    cudaFree(ws);
    return rc;  /* u32scan_strerror(rc) names a failure */
}

/* With an argument: scan 2^20 ones on the default stream (needs a GPU). */
int main(int argc, char **argv)
{
    (void)argv;
    if (argc < 2) return 0;
    const size_t n = (size_t)1 << 20;
    uint32_t *d = NULL, *total = NULL;
    if (cudaMalloc((void **)&d, 4 * n) != cudaSuccess || cudaMalloc((void **)&total, 4) != cudaSuccess) return 1;
    if (cudaMemset(d, 0, 4 * n) != cudaSuccess) return 1;
    int rc = scan_in_place(d, n, total, 0);
    cudaFree(d);
    cudaFree(total);
    return rc == U32SCAN_OK ? 0 : 1;
}

// inputs.cu -- the seeded synthetic inputs, drawn on the device.
//
// Counter-based SplitMix64 (S. Vigna's public-domain mixer, the output
// function of java.util.SplittableRandom), the definition the host
// generator (u32_prefix_scan_gb300/inputs.py) follows: element i of stream
// `stream` under seed `seed` is the high half of
//
//   z = ((seed << 40) | (stream << 32) | i) + 0x9E3779B97F4A7C15
//   z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
//   z = (z ^ (z >> 27)) * 0x94D049BB133111EB
//   z =  z ^ (z >> 31)                                  (all mod 2^64)
//
// Drawing a large input here spares a copy of it from the host. This file
// draws numbers only: none of the library's operations use it.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace u32scan {

__global__ void __launch_bounds__(256)
fill_splitmix_kernel(uint32_t *__restrict__ out, unsigned long long n, unsigned long long base,
                     unsigned long long start) {
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        unsigned long long z = (base | (start + i)) + 0x9E3779B97F4A7C15ull;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        out[i] = (uint32_t)(z >> 32);
    }
}

static std::mutex g_fill_mu;
static int g_fill_sms[64];

}  // namespace u32scan

using namespace u32scan;

extern "C" int u32scan_fill_splitmix_u32(uint32_t *out, size_t n, uint32_t seed, uint32_t stream, size_t start,
                                         u32scan_stream_t s) {
    if (n == 0) return U32SCAN_OK;
    if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 3) || seed >= (1u << 24) || stream >= 256u ||
        start >= (1ull << 32) || n > (1ull << 32) - start)
        return U32SCAN_EINVAL;
    int dev = -1, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return U32SCAN_ECUDA;
    {
        std::lock_guard<std::mutex> lock(g_fill_mu);
        if (g_fill_sms[dev] == 0 &&
            cudaDeviceGetAttribute(&g_fill_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return U32SCAN_ECUDA;
        sms = g_fill_sms[dev];
    }
    // eight resident blocks of 256 an SM, no more blocks than elements need
    const unsigned long long want = (n + 255) / 256;
    const unsigned int grid = want < (unsigned long long)(8 * sms) ? (unsigned int)want : (unsigned int)(8 * sms);
    const unsigned long long base = ((unsigned long long)seed << 40) | ((unsigned long long)stream << 32);
    fill_splitmix_kernel<<<grid, 256, 0, (cudaStream_t)s>>>(out, n, base, start);
    return cudaGetLastError() == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

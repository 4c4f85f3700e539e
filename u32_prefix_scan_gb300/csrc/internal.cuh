// internal.cuh -- device-side building blocks shared by the library's kernels.
//
// Single-pass tile carry ("decoupled look-back"): every tile of a kernel
// publishes, in one 64-bit word of the workspace, first its own aggregate
// and later its inclusive prefix (the sum of everything up to and including
// it). A tile finds its exclusive prefix by reading its predecessors' words
// 32 at a time, newest first, adding aggregates until it meets an inclusive
// prefix. This replaces the three-pass block-sums / base-scan / rescan scheme
// of the scan.bend page and the turn-passing relay of cubecl's Relay: the
// data is read once and written once (8 bytes per element for a scan).
//
// Forward progress: a tile's index comes from an atomic counter, not from
// blockIdx, so every predecessor of a running tile has already started
// (the hazard the Relay page names: a waiting block holds its place on the
// device). Every wait is bounded by a time limit read from %globaltimer;
// on expiry the tile records U32SCAN_ETIMEOUT in the workspace status word,
// stops waiting and finishes, so a kernel never hangs the GPU.
//
// Workspace: [header (256 B)] [tile words, 8 B each].
// Descriptors carry a tag derived from a per-workspace launch counter
// ("epoch"), so words left by earlier launches read as "not ready" and the
// workspace needs zeroing only once, before its first use. That holds as
// long as the workspace holds nothing but tile words at those offsets: the
// radix sort also keeps histograms and ping-pong buffers in the workspace
// (stale small integers there could pass for tagged words). A large sort
// keeps them past the span any other operation's tile words can occupy
// (tile_word_reach) and leaves only tagged words inside it; a small sort
// packs them after the header and clears that span before it returns.
//
// Re-arming. Every block reads the epoch before its first draw; the block
// that draws the launch's last index resets the tile counter and advances
// the epoch for the next launch (every other block has read the epoch
// before its own draw, and the draw is an acq_rel RMW, so none can see the
// new epoch). A tag holds 29 bits of the epoch, so tags repeat every 2^29
// launches. Every block knows from its epoch whether its launch is the last
// of a tag period; in that launch alone the blocks count themselves out as
// they finish (finish_period), and the last one out zeroes the tile words,
// so no word from the period that ends can pass for a word of the next one.
// Other launches pay nothing for this. (A launch whose blocks stop early on
// a bulk-copy timeout may leave the tile counter unreset; the timeout is
// reported, and the workspace must be zero-filled again before reuse.)
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "u32scan.h"

namespace u32scan {

struct WsHeader {
    unsigned int counter;   // next tile index to hand out
    unsigned int epoch;     // call generation
    unsigned int status;    // device-side error bits (kStatus*)
    unsigned int detail;    // first tile that timed out, + 1 (0 = none)
    unsigned int done;      // blocks of the running launch that have finished
    unsigned int pad0[27];
    unsigned long long seg_count;  // segmented scans: tiles counted and heads (byte 128, its own line)
    unsigned int pad1[30];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

constexpr size_t kHeaderBytes = 256;
constexpr unsigned int kStatusTimeout = 1u;
constexpr unsigned long long kDefaultLimitNs = 1000000000ull;  // 1 s
constexpr unsigned int kMaxSpinIters = 1u << 24;

// Tile word layout: bits 0..31 value, bit 32 P (inclusive prefix, else
// aggregate), bit 33 H (segmented: a head lies in the summed range),
// bits 34..63 tag (never 0 for a published word).
constexpr unsigned long long kFlagP = 1ull << 32;
constexpr unsigned long long kFlagH = 1ull << 33;
constexpr unsigned long long kTagMask = ~((1ull << 34) - 1ull);

__host__ __device__ inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Clear workspace bytes on `stream` (see the workspace note above).
static inline int clear_tile_words(void *p, size_t bytes, cudaStream_t stream) {
    return cudaMemsetAsync(p, 0, bytes, stream) == cudaSuccess ? U32SCAN_OK : U32SCAN_ECUDA;
}

// Launches per tag period: tag_of(e) == tag_of(e + kTagPeriod).
constexpr unsigned int kTagPeriod = 1u << 29;

__device__ __forceinline__ unsigned long long tag_of(unsigned int epoch) {
    return (unsigned long long)((epoch & (kTagPeriod - 1u)) + 1u) << 34;
}

__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned int *p, unsigned int v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned int atom_add_acq_rel(unsigned int *p, unsigned int v) {
    unsigned int r;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(r) : "l"(p), "r"(v) : "memory");
    return r;
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Draw this block's tile index (thread 0 only). Returns the index and the
// epoch of this call; the block drawing index n_tiles - 1 re-arms the header.
// (One 64-bit atomic returning counter and epoch together measured 2 %
// slower in the radix digit pass than this load and 32-bit add.)
__device__ __forceinline__ unsigned int draw_tile(WsHeader *hdr, unsigned int n_tiles,
                                                  unsigned int *epoch_out) {
    const unsigned int e = ld_relaxed_u32(&hdr->epoch);
    const unsigned int t = atom_add_acq_rel(&hdr->counter, 1u);
    if (t == n_tiles - 1u) {
        st_relaxed_u32(&hdr->counter, 0u);
        st_relaxed_u32(&hdr->epoch, e + 1u);
    }
    *epoch_out = e;
    return t;
}

// The end of a tag period (all threads of every block call it, once, after
// the block's last access to the workspace; a no-op unless this launch,
// epoch `epoch`, is the period's last). Then each block counts itself out,
// and the last one out zeroes the first `clear_words` tile words (`words`:
// the tile words after the header), which must cover every tile word a
// later launch on this workspace can read.
__device__ __forceinline__ void finish_period(WsHeader *hdr, unsigned int epoch, unsigned long long *words,
                                              unsigned long long clear_words) {
    if (((epoch + 1u) & (kTagPeriod - 1u)) != 0u || clear_words == 0ull) return;  // the same in every block
    __shared__ unsigned int s_last_out;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const bool last = atom_add_acq_rel(&hdr->done, 1u) == gridDim.x - 1u;
        if (last) st_relaxed_u32(&hdr->done, 0u);
        s_last_out = last ? 1u : 0u;
    }
    __syncthreads();
    if (s_last_out)
        for (unsigned long long i = threadIdx.x; i < clear_words; i += blockDim.x) words[i] = 0ull;
}

__device__ __forceinline__ void report_timeout(WsHeader *hdr, unsigned int tile) {
    atomicOr(&hdr->status, kStatusTimeout);
    atomicCAS(&hdr->detail, 0u, tile + 1u);
}

// Inclusive warp scan (wrapping u32 sums).
__device__ __forceinline__ unsigned int warp_inclusive_sum(unsigned int x, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        unsigned int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    return x;
}

// ---------------------------------------------------------------------------
// The scans' operators: the integer operators of the CAIRN "Concurrency"
// page's reduce and scan (add_wrap, mul_wrap, &, |, ^, min, max), on u32.
// Each is associative and commutative, so a look-back may combine words in
// any order.
// ---------------------------------------------------------------------------
enum MonoidCode { kAdd = 0, kMul = 1, kAnd = 2, kOr = 3, kXor = 4, kMin = 5, kMax = 6 };

template <int OP>
struct Monoid {
    static __device__ __forceinline__ unsigned int identity() {
        return OP == kMul ? 1u : (OP == kAnd || OP == kMin) ? 0xffffffffu : 0u;
    }
    static __device__ __forceinline__ unsigned int apply(unsigned int a, unsigned int b) {
        switch (OP) {
        case kAdd: return a + b;
        case kMul: return a * b;
        case kAnd: return a & b;
        case kOr: return a | b;
        case kXor: return a ^ b;
        case kMin: return a < b ? a : b;
        default: return a > b ? a : b;
        }
    }
    // Fold of the 32 lanes' values (all lanes get it).
    static __device__ __forceinline__ unsigned int warp_fold(unsigned int v) {
        switch (OP) {
        case kAdd: return __reduce_add_sync(0xffffffffu, v);
        case kAnd: return __reduce_and_sync(0xffffffffu, v);
        case kOr: return __reduce_or_sync(0xffffffffu, v);
        case kXor: return __reduce_xor_sync(0xffffffffu, v);
        case kMin: return __reduce_min_sync(0xffffffffu, v);
        case kMax: return __reduce_max_sync(0xffffffffu, v);
        default:
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) v = apply(v, __shfl_xor_sync(0xffffffffu, v, d));
            return v;
        }
    }
    // Inclusive scan across the lanes of a warp.
    static __device__ __forceinline__ unsigned int warp_inclusive(unsigned int x, int lane) {
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned int y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x = apply(y, x);
        }
        return x;
    }
    // The lane's exclusive value given its inclusive one and its own input.
    static __device__ __forceinline__ unsigned int warp_exclusive(unsigned int inc, unsigned int own, int lane) {
        if (OP == kAdd) return inc - own;
        const unsigned int prev = __shfl_up_sync(0xffffffffu, inc, 1);
        return lane == 0 ? identity() : prev;
    }
};

// Split form of the wide look-back for software-pipelined blocks, which
// publish a tile's aggregate as soon as it is known and walk its look-back
// one tile later: publish_aggregate, then lookback_prefix_wide, then
// publish_inclusive. Tile 0's aggregate is its inclusive prefix at once.
__device__ __forceinline__ void publish_aggregate(unsigned long long *desc, unsigned int t, unsigned int agg,
                                                  unsigned long long tag) {
    st_relaxed(desc + t, tag | (t == 0 ? kFlagP : 0ull) | agg);
}

__device__ __forceinline__ void publish_inclusive(unsigned long long *desc, unsigned int t, unsigned int incl,
                                                  unsigned long long tag) {
    st_relaxed(desc + t, tag | kFlagP | incl);
}

// First look-back window of tile t: word j of lane l is the carry word of
// the tile 32 * j + l + 1 places back (a virtual inclusive prefix holding
// the operator's identity before tile 0).
// Loading it early lets its L2 round trip overlap other work.
// (STRIDE: words between consecutive tiles' words, for descriptors that
// interleave several words a tile.)
template <int K, int OP = kAdd, int STRIDE = 1>
__device__ __forceinline__ void lookback_window(const unsigned long long *desc, long long pos,
                                                unsigned long long tag, int lane, unsigned long long (&d)[K]) {
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const long long idx = pos - 32 * j - lane;
        d[j] = idx >= 0 ? ld_relaxed(desc + STRIDE * idx) : (tag | kFlagP | Monoid<OP>::identity());
    }
}

// Fold (under OP) of tiles 0 .. t-1 (all 32 lanes call it), starting from a
// first window `d` already loaded by lookback_window(desc, t - 1, ...).
// Stops at (and includes) the nearest word with a STOP flag (the inclusive
// prefix, kFlagP, by default); a round needs readiness only up to there, so
// slow far-away words are never waited for.
template <int K, int OP = kAdd, int STRIDE = 1, unsigned long long STOP = kFlagP>
__device__ __forceinline__ unsigned int lookback_prefix_wide(const unsigned long long *desc, unsigned int t,
                                                             unsigned long long tag, WsHeader *hdr,
                                                             unsigned long long limit_ns, int lane,
                                                             unsigned long long (&d)[K]) {
    using M = Monoid<OP>;
    if (t == 0) return M::identity();
    unsigned int prefix = M::identity();
    long long pos = (long long)t - 1;
    while (true) {
        unsigned long long t0 = 0;
        for (unsigned int iter = 0;; ++iter) {
            // Distance order: word j of lane l is 32 * j + l + 1 tiles back.
            // Find the first word (in that order) that is either not ready
            // or an inclusive prefix.
            int stop_j = K, stop_lane = 0;
            bool stop_ready = true;
#pragma unroll
            for (int j = K - 1; j >= 0; --j) {
                const bool ready = (d[j] & kTagMask) == tag;
                const unsigned int m = __ballot_sync(0xffffffffu, !ready || (d[j] & STOP));
                if (m) {
                    stop_j = j;
                    stop_lane = __ffs(m) - 1;
                    stop_ready = (__shfl_sync(0xffffffffu, ready ? 1u : 0u, stop_lane) != 0);
                }
            }
            if (stop_j == K) {  // whole window ready, no inclusive prefix: fold it all, move back
                unsigned int sum = M::identity();
#pragma unroll
                for (int j = 0; j < K; ++j) sum = M::apply(sum, (unsigned int)d[j]);
                prefix = M::apply(prefix, M::warp_fold(sum));
                break;
            }
            if (stop_ready) {  // an inclusive prefix with everything nearer ready: done
                unsigned int sum = M::identity();
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (j < stop_j || (j == stop_j && lane <= stop_lane)) sum = M::apply(sum, (unsigned int)d[j]);
                prefix = M::apply(prefix, M::warp_fold(sum));
                return prefix;
            }
            // A nearer word is not ready yet: reload the words not ready.
            if (iter == 0) t0 = __shfl_sync(0xffffffffu, globaltimer(), 0);
            if (iter >= 8) __nanosleep(32);
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const long long idx = pos - 32 * j - lane;
                if (idx >= 0 && (d[j] & kTagMask) != tag) d[j] = ld_relaxed(desc + STRIDE * idx);
            }
            const unsigned long long now = __shfl_sync(0xffffffffu, globaltimer(), 0);
            if (iter > 0 && (now - t0 > limit_ns || iter >= kMaxSpinIters)) {
                if (lane == 0) report_timeout(hdr, t);
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if ((d[j] & kTagMask) != tag) d[j] = tag | kFlagP | M::identity();
            }
        }
        pos -= 32 * K;
        lookback_window<K, OP, STRIDE>(desc, pos, tag, lane, d);
    }
}

// ---------------------------------------------------------------------------
// Segmented scans carry two words per tile (at desc2 + 2 * tile):
//   word A  the segmented carry: value = sum since the last head in the
//           summed range; kFlagH when that range holds a head (the value is
//           then complete on its own); kFlagP when it is the final value at
//           the tile's end;
//   word B  the running head count (plain sum), kFlagP when final.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned int lanemask_le(int lane) { return 0xffffffffu >> (31 - lane); }
__device__ __forceinline__ unsigned int lanemask_lt(int lane) { return (1u << lane) - 1u; }

// Segmented inclusive scan across the lanes of a warp. Lane l holds the
// segmented sum of its own run (`t`: the sum since its last head, or of the
// whole run when `has_head` is false); `carry` is the segmented value before
// lane 0. Returns the segmented value at the end of lane l's run. With P the
// plain inclusive scan of t and L the last lane at or before l holding a
// head, that value is P[l] - P[L-1] (or carry + P[l] when there is no L).
__device__ __forceinline__ unsigned int warp_segmented_inclusive(unsigned int t, bool has_head, unsigned int carry,
                                                                 int lane) {
    const unsigned int P = warp_inclusive_sum(t, lane);
    const unsigned int m = __ballot_sync(0xffffffffu, has_head) & lanemask_le(lane);
    const int L = 31 - __clz(m | 1u);  // (m | 1) keeps the index valid; unused when m == 0
    const unsigned int before_L = __shfl_sync(0xffffffffu, P - t, L);
    return m ? P - before_L : carry + P;
}

struct SegPrefix {
    unsigned int seg;  // segmented value just before the tile
    unsigned int cnt;  // heads before the tile
};


// Both look-backs of tile t (all 32 lanes call it), each with the library's
// windowed walk: word A
// (stops at a word with a head or a final value) KA, word B (stops at a
// final count) KB words a lane per round trip; both first windows are in
// flight together. Word A usually stops one tile back (tiles that hold a
// head); word B walks to the nearest tile whose count is final, which with
// every SM's tiles in flight can be a block's worth of tiles back.
template <int KA, int KB>
__device__ __forceinline__ SegPrefix lookback_seg_wide(const unsigned long long *desc2, unsigned int t,
                                                       unsigned long long tag, WsHeader *hdr,
                                                       unsigned long long limit_ns, int lane) {
    SegPrefix pre{0u, 0u};
    if (t == 0) return pre;
    unsigned long long wa[KA], wb[KB];
    lookback_window<KA, kAdd, 2>(desc2, (long long)t - 1, tag, lane, wa);
    lookback_window<KB, kAdd, 2>(desc2 + 1, (long long)t - 1, tag, lane, wb);
    pre.seg = lookback_prefix_wide<KA, kAdd, 2, kFlagP | kFlagH>(desc2, t, tag, hdr, limit_ns, lane, wa);
    pre.cnt = lookback_prefix_wide<KB, kAdd, 2, kFlagP>(desc2 + 1, t, tag, hdr, limit_ns, lane, wb);
    return pre;
}

// ---------------------------------------------------------------------------
// Shared-memory staging with the Tensor Memory Accelerator's bulk copy
// (cp.async.bulk, 1-D: 16-byte aligned addresses, size a multiple of 16)
// completing on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned int smem_u32(const void *p) {
    return static_cast<unsigned int>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned int bar, unsigned int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses (and, after a block
// barrier, those of the block) before later async-proxy (bulk copy) ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned int bar, unsigned int bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned int bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned int bar, unsigned int parity) {
    unsigned int done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

// Wait for phase `parity` of the barrier to complete, bounded by limit_ns
// (and an iteration cap). Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned int bar, unsigned int parity,
                                                  unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (unsigned int iter = 0; iter < kMaxSpinIters; ++iter) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
    return false;
}

__device__ __forceinline__ void bulk_load(unsigned int dst_smem, const void *src, unsigned int bytes,
                                          unsigned int bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst_smem),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Ask for `bytes` at `src` (16-byte aligned, a multiple of 16) to be brought
// into L2, without waiting.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, unsigned int bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Shared memory -> global 1-D bulk copy (16-byte aligned, size a multiple of
// 16), tracked as a bulk-async group of the issuing thread.
__device__ __forceinline__ void bulk_store(void *dst, unsigned int src_smem, unsigned int bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until this thread's bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until this thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tile words (8 bytes each, after the header) that the last launch of a tag
// period zeroes in a workspace of ws_bytes: all of them, up to the largest
// span any operation's tile words can take (defined in api.cu).
unsigned long long tile_words_to_clear(size_t ws_bytes);
size_t tile_word_reach();

// Host-side workspace sizing of each operation (defined beside its kernels).
size_t scan_workspace_bytes(unsigned long long n);
size_t scan_workspace_bytes_upto(unsigned long long m);
size_t scan_host_workspace_bytes(unsigned long long n);
size_t segscan_workspace_bytes(unsigned long long n);
size_t compact_workspace_bytes(unsigned long long n);
size_t radix_workspace_bytes(unsigned long long n);
size_t compact_values_workspace_bytes(unsigned long long n);
size_t scan64_workspace_bytes(unsigned long long n);
size_t reduce_workspace_bytes();

// In-library launches of the add-scan: one chunk of a longer array after a
// device carry-in (the host-buffer pipeline), and the inclusive scan with
// its total (the runs layout).
int scan_chunk_launch(bool inclusive, uint32_t *data, unsigned long long n, const uint32_t *carry_in,
                      uint32_t *total, void *ws, size_t ws_bytes, cudaStream_t stream);
int scan_inclusive_launch(uint32_t *data, unsigned long long n, uint32_t *total, void *ws, size_t ws_bytes,
                          cudaStream_t stream);

}  // namespace u32scan

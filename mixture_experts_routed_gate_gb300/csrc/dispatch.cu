// dispatch.cu -- the counting-sort dispatch of the routed MoE forward.
//
// CSDN "forward", steps 2-5 (argsort by expert, bincount, cumsum, the
// per-expert gather loop, group_sizes / group_offset / group_padded_offsets /
// group_idx_for_bx) done on the device with no host round trip:
//   1. dispatch_hist_kernel: each CTA counts the experts of its chunk of
//      CHUNK consecutive pairs (f = t*k + j) into hist[chunk][e].
//   2. dispatch_scan_scatter_kernel, one CTA per chunk: each CTA sums the
//      chunk histograms itself (per-expert totals and its chunk's bases), two
//      block scans give group_offsets and the padded offsets, a binary search
//      per M block gives group_idx_for_bx (spread over the CTAs; CTA 0 writes
//      the per-expert tables); then warp-level counts in shared memory give
//      every warp its start per expert, and the warp walks its pairs 32 at a
//      time in ascending f, ranking equal experts with __match_any_sync, so
//      the order inside an expert is ascending f (a stable sort) with no
//      atomics-order effects.
// Problems of at most 16384 pairs and 256 experts run all of it in a single
// CTA (dispatch_small_kernel): one launch instead of two.
#include <mutex>

#include "../../include/moe_routed_gate.h"
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int DS_WARPS = 8;
constexpr int DS_THREADS = DS_WARPS * 32;
constexpr int PAIRS_PER_WARP = 256;
constexpr int CHUNK = DS_WARPS * PAIRS_PER_WARP;  // 2048 pairs per CTA

__global__ void __launch_bounds__(DS_THREADS)
    dispatch_hist_kernel(const int32_t *__restrict__ idx, int64_t n_pairs, int E,
                         int32_t *__restrict__ hist) {
    extern __shared__ int32_t counts[];
    for (int e = threadIdx.x; e < E; e += DS_THREADS) counts[e] = 0;
    griddep_wait();
    griddep_launch_dependents();
    __syncthreads();
    const int64_t f0 = static_cast<int64_t>(blockIdx.x) * CHUNK;
    // all of the thread's loads first, then the counts
    constexpr int PER_THREAD = CHUNK / DS_THREADS;
    int ev[PER_THREAD];
#pragma unroll
    for (int i = 0; i < PER_THREAD; ++i) {
        const int64_t f = f0 + i * DS_THREADS + threadIdx.x;
        ev[i] = f < n_pairs ? __ldg(idx + f) : -1;
    }
#pragma unroll
    for (int i = 0; i < PER_THREAD; ++i)
        if (ev[i] >= 0 && ev[i] < E) atomicAdd(&counts[ev[i]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += DS_THREADS)
        hist[static_cast<int64_t>(blockIdx.x) * E + e] = counts[e];
}

// Exclusive scan of one value per thread over the whole block (<= 1024 threads).
__device__ int block_exclusive_scan(int v, int *warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, s);
        if (lane >= s) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        int ws = lane < nw ? warp_sums[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, s);
            if (lane >= s) wi += o;
        }
        warp_sums[lane] = wi - ws;  // exclusive prefix of warp totals
    }
    __syncthreads();
    const int out = warp_sums[warp] + incl - v;
    __syncthreads();  // warp_sums is reused by the next call
    return out;
}

// Steps 2 and 3 in one launch: every CTA sums the raw chunk histograms
// itself (its chunk's per-expert bases, the group sizes and both block
// scans), so no separate scan grid runs between the histogram and the
// scatter.  CTA 0 writes sizes / offsets / padded; the M-block lookup and the
// expert MLP's counters are spread over the CTAs.
constexpr int DS_MAX_PER_THREAD = 4;  // E <= 4 * DS_THREADS = 1024

__global__ void __launch_bounds__(DS_THREADS)
    dispatch_scan_scatter_kernel(const int32_t *__restrict__ idx, const float *__restrict__ w,
                                 int64_t n_pairs, int k, int E, int block_m, const int32_t *__restrict__ hist,
                                 int n_chunks, int32_t *__restrict__ sizes, int32_t *__restrict__ offsets,
                                 int32_t *__restrict__ padded, int32_t *__restrict__ gidx, int m_blocks,
                                 int32_t *__restrict__ ready, int32_t *__restrict__ sorted_tok,
                                 float *__restrict__ sorted_w, int32_t *__restrict__ pos) {
    extern __shared__ int32_t ds_smem[];
    int32_t *wcount = ds_smem;                  // [DS_WARPS][E]
    int32_t *po_s = ds_smem + DS_WARPS * E;     // [E] padded offsets
    int32_t *cbase = po_s + E;                  // [E] this chunk's first row per expert
    __shared__ int warp_sums[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < DS_WARPS * E; i += DS_THREADS) wcount[i] = 0;
    griddep_wait();
    griddep_launch_dependents();
    // this warp's pairs (expert ids and weights) in registers, loaded once
    // and before the histogram sums so that both latencies overlap
    constexpr int ROUNDS = PAIRS_PER_WARP / 32;
    const int64_t wf0 = static_cast<int64_t>(blockIdx.x) * CHUNK + static_cast<int64_t>(warp) * PAIRS_PER_WARP;
    int ev[ROUNDS];
    float wv[ROUNDS];
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int64_t f = wf0 + r * 32 + lane;
        int e = f < n_pairs ? __ldg(idx + f) : -1;
        ev[r] = (e >= 0 && e < E) ? e : -1;
        wv[r] = (w && f < n_pairs) ? __ldg(w + f) : 1.0f;
    }
    // totals and this chunk's bases of the experts e = per * tid + i
    const int per = (E + DS_THREADS - 1) / DS_THREADS;
    int tot[DS_MAX_PER_THREAD], bas[DS_MAX_PER_THREAD];
    int my_tot = 0, my_pad = 0;
#pragma unroll
    for (int i = 0; i < DS_MAX_PER_THREAD; ++i) {
        const int e = threadIdx.x * per + i;
        tot[i] = 0;
        bas[i] = 0;
        if (i < per && e < E) {
#pragma unroll 4
            for (int c = 0; c < n_chunks; ++c) {
                const int v = hist[static_cast<int64_t>(c) * E + e];
                if (c < static_cast<int>(blockIdx.x)) bas[i] += v;
                tot[i] += v;
            }
            my_tot += tot[i];
            // padded size of expert e: ceil((count + 1) / block_m) * block_m
            my_pad += ((tot[i] + block_m) / block_m) * block_m;
        }
    }
    int run = block_exclusive_scan(my_tot, warp_sums);
    int prun = block_exclusive_scan(my_pad, warp_sums);
#pragma unroll
    for (int i = 0; i < DS_MAX_PER_THREAD; ++i) {
        const int e = threadIdx.x * per + i;
        if (i < per && e < E) {
            if (blockIdx.x == 0) {
                sizes[e] = tot[i];
                offsets[e] = run;
                padded[e] = prun;
            }
            po_s[e] = prun;
            cbase[e] = run + bas[i];
            run += tot[i];
            prun += ((tot[i] + block_m) / block_m) * block_m;
        }
    }
    __syncthreads();
    // group_idx_for_bx[bx] = last e with bx * block_m >= po[e] (po[0] = 0, increasing)
    for (int bx = blockIdx.x * DS_THREADS + threadIdx.x; bx < m_blocks; bx += gridDim.x * DS_THREADS) {
        const long long start = static_cast<long long>(bx) * block_m;
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<long long>(po_s[mid]) <= start) lo = mid;
            else hi = mid - 1;
        }
        gidx[bx] = lo;
        if (ready) ready[bx] = 0;
    }
    if (ready && blockIdx.x == 0 && threadIdx.x == 0) ready[m_blocks] = 0;  // the expert MLP's tile counter

    int32_t *mine = wcount + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    // pass 1: per-warp expert counts
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const unsigned peers = __match_any_sync(0xffffffffu, ev[r]);
        if (ev[r] >= 0 && (peers & lt_mask) == 0) mine[ev[r]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // warp starts per expert: chunk base + counts of the earlier warps
    for (int e = threadIdx.x; e < E; e += DS_THREADS) {
        int r0 = cbase[e];
        for (int wv = 0; wv < DS_WARPS; ++wv) {
            const int c = wcount[wv * E + e];
            wcount[wv * E + e] = r0;
            r0 += c;
        }
    }
    __syncthreads();
    // pass 2: stable ranks inside the warp, 32 pairs at a time in ascending f
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int64_t f = wf0 + r * 32 + lane;
        const int e = ev[r];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int row = 0;
        if (e >= 0) row = mine[e] + __popc(peers & lt_mask);
        __syncwarp();
        if (e >= 0 && (peers & lt_mask) == 0) mine[e] += __popc(peers);  // lowest peer updates
        __syncwarp();
        if (e >= 0) {
            sorted_tok[row] = static_cast<int32_t>(f / k);
            sorted_w[row] = wv[r];
            pos[f] = row;
        }
    }
}

// Whole dispatch in one CTA for small problems (at most SMALL_MAX_PAIRS pairs
// and SMALL_MAX_E experts): the pairs stay in registers (warp w owns a
// contiguous run of 32*R pairs), per-warp counts in shared memory, one block
// scan, the block lookup, then the stable scatter from the same registers.
constexpr int SMALL_MAX_ROUNDS = 16;
constexpr int SMALL_MAX_PAIRS = 1024 * SMALL_MAX_ROUNDS;  // 16384
constexpr int SMALL_MAX_E = 256;

template <int SMALL_THREADS>
__global__ void __launch_bounds__(SMALL_THREADS)
    dispatch_small_kernel(const int32_t *__restrict__ idx, const float *__restrict__ w,
                          int n_pairs, int k, int E, int block_m, int32_t *__restrict__ sizes,
                          int32_t *__restrict__ offsets, int32_t *__restrict__ padded,
                          int32_t *__restrict__ gidx, int m_blocks,
                          int32_t *__restrict__ sorted_tok, float *__restrict__ sorted_w,
                          int32_t *__restrict__ pos, int32_t *__restrict__ ready) {
    constexpr int SMALL_WARPS = SMALL_THREADS / 32;
    static_assert(SMALL_THREADS >= SMALL_MAX_E, "one thread per expert");
    __shared__ int32_t wcount[SMALL_WARPS * SMALL_MAX_E];
    __shared__ int po_s[SMALL_MAX_E];
    __shared__ int warp_sums[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rounds = (n_pairs + SMALL_THREADS - 1) / SMALL_THREADS;  // <= SMALL_MAX_ROUNDS
    const int wf0 = warp * rounds * 32;
    for (int i = threadIdx.x; i < SMALL_WARPS * E; i += SMALL_THREADS) wcount[i] = 0;
    // release the next kernel before waiting: its CTAs become resident while
    // the gate still runs and start their own independent set-up (every
    // dependent waits for this grid before it reads the tables)
    griddep_launch_dependents();
    griddep_wait();
    int ev[SMALL_MAX_ROUNDS];
#pragma unroll
    for (int r = 0; r < SMALL_MAX_ROUNDS; ++r) {
        const int f = wf0 + r * 32 + lane;
        int e = -1;
        if (r < rounds && f < n_pairs) e = __ldg(idx + f);
        ev[r] = (e >= 0 && e < E) ? e : -1;
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    int32_t *mine = wcount + warp * E;
#pragma unroll
    for (int r = 0; r < SMALL_MAX_ROUNDS; ++r) {
        if (r < rounds) {
            const unsigned peers = __match_any_sync(0xffffffffu, ev[r]);
            if (ev[r] >= 0 && (peers & lt_mask) == 0) mine[ev[r]] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    const int e = threadIdx.x;
    int count = 0;
    if (e < E) {
        for (int wv = 0; wv < SMALL_WARPS; ++wv) {
            const int c = wcount[wv * E + e];
            wcount[wv * E + e] = count;
            count += c;
        }
    }
    const int off = block_exclusive_scan(e < E ? count : 0, warp_sums);
    const int psize = e < E ? ((count + block_m) / block_m) * block_m : 0;
    const int poff = block_exclusive_scan(psize, warp_sums);
    if (e < E) {
        sizes[e] = count;
        offsets[e] = off;
        padded[e] = poff;
        po_s[e] = poff;
        for (int wv = 0; wv < SMALL_WARPS; ++wv) wcount[wv * E + e] += off;
    }
    __syncthreads();
    for (int bx = threadIdx.x; bx < m_blocks; bx += SMALL_THREADS) {
        const long long start = static_cast<long long>(bx) * block_m;
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<long long>(po_s[mid]) <= start) lo = mid;
            else hi = mid - 1;
        }
        gidx[bx] = lo;
        if (ready) ready[bx] = 0;
    }
    if (ready && threadIdx.x == 0) ready[m_blocks] = 0;  // the expert MLP's tile counter
#pragma unroll
    for (int r = 0; r < SMALL_MAX_ROUNDS; ++r) {
        if (r < rounds) {
            const int f = wf0 + r * 32 + lane;
            const int ee = ev[r];
            const unsigned peers = __match_any_sync(0xffffffffu, ee);
            int row = 0;
            if (ee >= 0) row = mine[ee] + __popc(peers & lt_mask);
            __syncwarp();
            if (ee >= 0 && (peers & lt_mask) == 0) mine[ee] += __popc(peers);
            __syncwarp();
            if (ee >= 0) {
                sorted_tok[row] = f / k;
                sorted_w[row] = w ? __ldg(w + f) : 1.0f;
                pos[f] = row;
            }
        }
    }
}

}  // namespace

size_t dispatch_scratch_bytes(int64_t n_pairs, int64_t E) {
    const int64_t n_chunks = n_pairs > 0 ? (n_pairs + CHUNK - 1) / CHUNK : 1;
    return static_cast<size_t>(n_chunks * E * 4);
}

cudaError_t launch_dispatch(const int32_t *topk_idx, const float *topk_w, int64_t T, int64_t k,
                            int64_t E, int64_t block_m, int32_t *sizes, int32_t *offsets, int32_t *padded,
                            int32_t *gidx, int64_t m_blocks, int32_t *sorted_token_idx,
                            float *sorted_row_weight, int32_t *pos, void *scratch,
                            int32_t *ready, cudaStream_t stream) {
    const int64_t n_pairs = T * k;
    if (n_pairs <= SMALL_MAX_PAIRS && E <= SMALL_MAX_E) {
        // fewer threads (shorter per-expert walks and scans) for few pairs
        auto kern = n_pairs <= 256 * SMALL_MAX_ROUNDS ? dispatch_small_kernel<256>
                                                      : dispatch_small_kernel<1024>;
        const int threads = n_pairs <= 256 * SMALL_MAX_ROUNDS ? 256 : 1024;
        return launch_pdl(kern, dim3(1), dim3(threads), 0, stream, topk_idx, topk_w,
                          static_cast<int>(n_pairs), static_cast<int>(k), static_cast<int>(E),
                          static_cast<int>(block_m), sizes, offsets, padded, gidx,
                          static_cast<int>(m_blocks), sorted_token_idx, sorted_row_weight, pos, ready);
    }
    const int64_t n_chunks = n_pairs > 0 ? (n_pairs + CHUNK - 1) / CHUNK : 0;
    int32_t *hist = static_cast<int32_t *>(scratch);
    if (n_chunks > 0) {
        cudaError_t e = launch_pdl(dispatch_hist_kernel, dim3(static_cast<unsigned>(n_chunks)),
                                   dim3(DS_THREADS), static_cast<size_t>(E * 4), stream, topk_idx,
                                   n_pairs, static_cast<int>(E), hist);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = static_cast<size_t>(DS_WARPS + 2) * E * 4;
    static std::atomic<size_t> attr_bytes[64];  // zero-initialised; several host threads may launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (smem > 48 * 1024 && (dev < 0 || dev >= 64 || attr_bytes[dev] < smem)) {
        cudaError_t e = cudaFuncSetAttribute(dispatch_scan_scatter_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_bytes[dev] = smem;
    }
    // one CTA per chunk (one CTA writes the tables when there are no pairs)
    const unsigned grid = static_cast<unsigned>(n_chunks > 0 ? n_chunks : 1);
    return launch_pdl(dispatch_scan_scatter_kernel, dim3(grid), dim3(DS_THREADS), smem, stream, topk_idx, topk_w,
                      n_pairs, static_cast<int>(k), static_cast<int>(E), static_cast<int>(block_m),
                      static_cast<const int32_t *>(hist), static_cast<int>(n_chunks), sizes, offsets, padded,
                      gidx, static_cast<int>(m_blocks), ready, sorted_token_idx, sorted_row_weight, pos);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Dispatch with no caller-provided scratch (moe_build_dispatch_noalloc).
//
// For callers that may not allocate device memory at all: code running while
// a CUDA graph is being captured (cudaMalloc is not a capturable operation),
// and engines whose device memory is planned once up front by another runtime
// so that no call may allocate, or fail for lack of memory, in the middle of
// a step.  Their per-chunk expert histograms live in this fixed array instead
// of a workspace.  Every GPU that loads the library keeps the array until the
// process exits.
// ---------------------------------------------------------------------------
static constexpr int64_t kStaticScratchInts = 262144;  // 1 MiB of int32 counters
static __device__ __align__(256) int32_t g_dispatch_static_scratch[kStaticScratchInts];

static std::mutex g_static_scratch_mu;
static void *g_static_scratch_addr[64];  // last address seen per device id

extern "C" MOE_API moe_status_t moe_build_dispatch_noalloc(
    const int32_t *topk_idx, const float *topk_w, int64_t T, int64_t k, int64_t E,
    int64_t block_m, int32_t *group_sizes, int32_t *group_offsets,
    int32_t *group_padded_offsets, int32_t *group_idx_for_bx, int32_t *sorted_token_idx,
    float *sorted_row_weight, int32_t *token_topk_to_pos, moe_stream_t stream) {
    const int st = moe::check_dispatch_args(topk_idx, T, k, E, block_m, group_sizes, group_offsets,
                                            group_padded_offsets, group_idx_for_bx,
                                            sorted_token_idx, sorted_row_weight, token_topk_to_pos);
    if (st != MOE_OK) return static_cast<moe_status_t>(st);
    // the histograms need ceil(T*k / 2048) * E counters
    if (moe::dispatch_scratch_bytes(T * k, E) > sizeof(g_dispatch_static_scratch))
        return MOE_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return MOE_ERR_CUDA;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_scratch_mu);
        // Host code only sees a stand-in symbol: ask the runtime for the
        // array's address in the current context.  Outside a capture the
        // address is looked up on every call (a host-side table lookup), so a
        // context re-created by cudaDeviceReset is picked up; during a capture
        // the address of the last call outside one is used.
        if (cap == cudaStreamCaptureStatusNone || g_static_scratch_addr[dev] == nullptr) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_dispatch_static_scratch) != cudaSuccess || !addr)
                return MOE_ERR_CUDA;
            g_static_scratch_addr[dev] = addr;
        }
        scratch = g_static_scratch_addr[dev];
    }
    // The histogram kernel writes every counter the later kernels read, so the
    // array needs no clearing between calls.
    const int64_t m_blocks = (T * k + block_m - 1) / block_m + E;
    cudaError_t e = moe::launch_dispatch(topk_idx, topk_w, T, k, E, block_m, group_sizes,
                                         group_offsets, group_padded_offsets, group_idx_for_bx,
                                         m_blocks, sorted_token_idx, sorted_row_weight,
                                         token_topk_to_pos, scratch, nullptr, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

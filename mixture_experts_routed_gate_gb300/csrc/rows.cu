// rows.cu -- the two row-moving steps of the routed MoE forward: the gather of
// token rows into expert order and the moe_reduce_fused combine.
#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// ---------------------------------------------------------------------------
// gather: a_out[r, :] = x[sorted_token_idx[r], :]  (CSDN "forward", step 3)
// One warp per row, 16-byte vectors, 4 in flight per lane; the rows are
// stored with the evict-first hint, so the stream of output rows does not push
// the token rows (read up to k times) out of L2.
// ---------------------------------------------------------------------------
constexpr int GA_WARPS = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(GA_WARPS * 32)
    gather_rows_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ idx,
                       int64_t n_rows, int nvec, uint4 *__restrict__ out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * GA_WARPS + warp;
    griddep_wait();
    griddep_launch_dependents();
    if (r >= n_rows) return;
    const uint4 *src = x + static_cast<int64_t>(__ldg(idx + r)) * nvec;
    uint4 *dst = out + r * nvec;
    int v = lane;
    for (; v + 96 < nvec; v += 128) {
        const uint4 a = ld_stream(src + v), b = ld_stream(src + v + 32);
        const uint4 c = ld_stream(src + v + 64), d = ld_stream(src + v + 96);
        __stcs(dst + v, a);
        __stcs(dst + v + 32, b);
        __stcs(dst + v + 64, c);
        __stcs(dst + v + 96, d);
    }
    for (; v < nvec; v += 32) __stcs(dst + v, ld_stream(src + v));
}

// The same rows in token order, for the forward: token t's row is read once
// and written to each of its rows token_topk_to_pos[t, j] (j < k <= 32; a
// position outside [0, n_rows), a dropped pair, is skipped).  The result is
// the row-order gather's, but x is read from memory once however many
// experts a token went to.  One warp per token.
__global__ void __launch_bounds__(GA_WARPS * 32)
    scatter_rows_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ pos, int64_t T, int k,
                        int64_t n_rows, int nvec, uint4 *__restrict__ out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * GA_WARPS + warp;
    griddep_wait();
    griddep_launch_dependents();
    if (t >= T) return;
    int p = -1;  // lane j < k: the row of slot j
    if (lane < k) {
        p = __ldg(pos + t * k + lane);
        if (p >= n_rows) p = -1;
    }
    const uint4 *src = x + t * nvec;
    for (int v = lane; v < nvec; v += 128) {
        uint4 a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (v + 32 * u < nvec) a[u] = ld_stream(src + v + 32 * u);
        for (int j = 0; j < k; ++j) {
            const int pj = __shfl_sync(0xffffffffu, p, j);
            if (pj < 0) continue;
            uint4 *dst = out + static_cast<int64_t>(pj) * nvec;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v + 32 * u < nvec) __stcs(dst + v + 32 * u, a[u]);
        }
    }
}

// The same scatter with the copy engine: a warp owns the tokens
// t = w, w + W, ... (W warps in the grid), which pass through two row buffers
// in shared memory.  Lane 0 loads a token's row with one bulk copy and writes
// it to each of its k rows with k bulk stores, the next token's load in
// flight meanwhile; the other lanes only read the positions.  A buffer is
// reloaded once the stores issued from it have read it.  Every wait is
// bounded: on expiry the warp records kErrTimeout, waits (bounded) for its
// loads in flight and stops.
// bounded wait for a copy still in flight (after a timeout): never hangs
__device__ __forceinline__ void rb_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long start = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - start > kWaitTimeoutNs) return;
}

constexpr int SB_MAX_WARPS = 4;
constexpr int SB_SMEM_BUDGET = 200 * 1024;

__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void bulk_s2g_hint(void *dst, uint32_t src, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(src), "r"(bytes), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(SB_MAX_WARPS * 32)
    scatter_rows_bulk_kernel(const uint8_t *__restrict__ x, const int32_t *__restrict__ pos, int64_t T, int k,
                             int64_t n_rows, uint32_t row_bytes, uint32_t buf_bytes, uint8_t *__restrict__ out,
                             int32_t *err) {
    extern __shared__ __align__(128) uint8_t sb_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const uint32_t buf = smem_u32(sb_smem) + static_cast<uint32_t>(warp) * 2u * buf_bytes;
    const uint32_t bar = smem_u32(sb_smem) + static_cast<uint32_t>(warps) * 2u * buf_bytes + warp * 16u;
    if (lane == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 8, 1);
        fence_mbar_init();
    }
    __syncwarp();
    griddep_wait();
    griddep_launch_dependents();
    const int64_t W = static_cast<int64_t>(gridDim.x) * warps;
    int64_t t = static_cast<int64_t>(blockIdx.x) * warps + warp;
    if (t >= T) return;
    const uint64_t pol = l2_policy_evict_first();
    volatile int abort_w = 0;
    if (lane == 0) {
        mbar_arrive_expect_tx(bar, row_bytes);
        bulk_g2s_hint(buf, x + t * row_bytes, row_bytes, bar, pol);
    }
    int p_next = lane < k ? __ldg(pos + t * k + lane) : -1;
    int64_t i = 0;
    bool ok = true;
    for (; t < T; t += W, ++i) {
        const uint32_t b = static_cast<uint32_t>(i & 1);
        const int p_cur = p_next;
        const int64_t tn = t + W;
        if (tn < T) {
            if (lane == 0) {
                bulk_wait_read_all();  // the other buffer's stores have read it
                mbar_arrive_expect_tx(bar + 8u * (b ^ 1u), row_bytes);
                bulk_g2s_hint(buf + (b ^ 1u) * buf_bytes, x + tn * row_bytes, row_bytes, bar + 8u * (b ^ 1u), pol);
            }
            p_next = lane < k ? __ldg(pos + tn * k + lane) : -1;
        }
        if (lane == 0) ok = mbar_wait_bounded(bar + 8u * b, static_cast<uint32_t>((i >> 1) & 1), &abort_w, err);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        for (int j = 0; j < k; ++j) {
            const int pj = __shfl_sync(0xffffffffu, p_cur, j);
            if (lane == 0 && pj >= 0 && pj < n_rows)
                bulk_s2g_hint(out + static_cast<int64_t>(pj) * row_bytes, buf + b * buf_bytes, row_bytes, pol);
        }
        if (lane == 0) bulk_commit();
    }
    if (lane == 0) {
        if (!ok) {
            // this token's load and, if issued, the next one's
            rb_wait_drain(bar + 8u * static_cast<uint32_t>(i & 1), static_cast<uint32_t>((i >> 1) & 1));
            if (t + W < T)
                rb_wait_drain(bar + 8u * static_cast<uint32_t>((i + 1) & 1),
                              static_cast<uint32_t>(((i + 1) >> 1) & 1));
        }
        bulk_wait_all();  // every store done before the buffers go away
    }
}

// ---------------------------------------------------------------------------
// copy: dst[i] = src[i] over 16-byte vectors, either side host memory the
// device can reach (pinned, mapped).  Every thread issues its loads before
// its stores, so a small copy costs one round trip over the host link.
// ---------------------------------------------------------------------------
constexpr int CP_THREADS = 256;
constexpr int CP_VEC = 4;  // vectors per thread per pass

// a plain (coherent) 16-byte load: the source may be host memory that the
// host wrote just before the launch, so not the read-only data path
__device__ __forceinline__ uint4 ld_coherent(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(CP_THREADS)
    copy_kernel(const uint4 *src, uint4 *__restrict__ dst, int64_t nvec) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * CP_THREADS;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * CP_THREADS + threadIdx.x; i0 < nvec;
         i0 += stride * CP_VEC) {
        uint4 v[CP_VEC];
#pragma unroll
        for (int j = 0; j < CP_VEC; ++j) {
            const int64_t i = i0 + j * stride;
            if (i < nvec) v[j] = ld_coherent(src + i);
        }
#pragma unroll
        for (int j = 0; j < CP_VEC; ++j) {
            const int64_t i = i0 + j * stride;
            if (i < nvec) dst[i] = v[j];
        }
    }
}

// ---------------------------------------------------------------------------
// moe_reduce_fused (TileOPs-Metax PR #55, section 1): one thread per 8
// consecutive hidden elements of one token.  The K slot rows are gathered
// with all loads of a group of 8 slots issued before any is consumed (the
// multi-slot look-ahead), then accumulated in ascending slot order in fp32 as
// acc = acc + (w * x), each product and sum rounded separately, padding
// slots (pos < 0) skipped, and the result cast once.  With that fixed order
// and rounding the result is the same bit pattern as the plain definition.
// ---------------------------------------------------------------------------
constexpr int RD_THREADS = 128;
constexpr int RD_LOOKAHEAD = 8;

template <typename TIn> struct Vec8;
template <> struct Vec8<__half> { uint4 v; };
template <> struct Vec8<__nv_bfloat16> { uint4 v; };
template <> struct Vec8<float> { uint4 a, b; };

template <typename TIn>
__device__ __forceinline__ Vec8<TIn> load8(const TIn *p);
template <>
__device__ __forceinline__ Vec8<__half> load8<__half>(const __half *p) {
    return Vec8<__half>{ld_stream(reinterpret_cast<const uint4 *>(p))};
}
template <>
__device__ __forceinline__ Vec8<__nv_bfloat16> load8<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return Vec8<__nv_bfloat16>{ld_stream(reinterpret_cast<const uint4 *>(p))};
}
template <>
__device__ __forceinline__ Vec8<float> load8<float>(const float *p) {
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    return Vec8<float>{ld_stream(q), ld_stream(q + 1)};
}

__device__ __forceinline__ void unpack8(const Vec8<__nv_bfloat16> &v, float (&f)[8]) {
    const uint32_t w[4] = {v.v.x, v.v.y, v.v.z, v.v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = unpack2<kBF16>(w[i]);
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}
__device__ __forceinline__ void unpack8(const Vec8<__half> &v, float (&f)[8]) {
    const uint32_t w[4] = {v.v.x, v.v.y, v.v.z, v.v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = unpack2<kF16>(w[i]);
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}
__device__ __forceinline__ void unpack8(const Vec8<float> &v, float (&f)[8]) {
    const uint32_t w[8] = {v.a.x, v.a.y, v.a.z, v.a.w, v.b.x, v.b.y, v.b.z, v.b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(w[i]);
}

template <typename TOut>
__device__ __forceinline__ void store8(TOut *p, const float (&f)[8]);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *p, const float (&f)[8]) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(pack2<kBF16>(f[0], f[1]), pack2<kBF16>(f[2], f[3]),
                                               pack2<kBF16>(f[4], f[5]), pack2<kBF16>(f[6], f[7]));
}
template <>
__device__ __forceinline__ void store8<__half>(__half *p, const float (&f)[8]) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(pack2<kF16>(f[0], f[1]), pack2<kF16>(f[2], f[3]),
                                               pack2<kF16>(f[4], f[5]), pack2<kF16>(f[6], f[7]));
}
template <>
__device__ __forceinline__ void store8<float>(float *p, const float (&f)[8]) {
    float4 *q = reinterpret_cast<float4 *>(p);
    q[0] = make_float4(f[0], f[1], f[2], f[3]);
    q[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// float8 e4m3fn output: round to nearest even, saturate to the finite range
template <>
__device__ __forceinline__ void store8<__nv_fp8_e4m3>(__nv_fp8_e4m3 *p, const float (&f)[8]) {
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        q[i] = __nv_cvt_float2_to_fp8x2(make_float2(f[2 * i], f[2 * i + 1]), __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<uint2 *>(p) = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(RD_THREADS)
    reduce_fused_kernel(const TIn *__restrict__ x, int64_t n_rows,
                        const int32_t *__restrict__ pos, const float *__restrict__ w,
                        const float *__restrict__ x_sf, const float *__restrict__ sf, int64_t T,
                        int K, int H, TOut *__restrict__ out, int32_t *__restrict__ err) {
    const int vpr = H >> 3;  // 8-element vectors per row
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * RD_THREADS + threadIdx.x;
    const int64_t t = gid / vpr;
    griddep_wait();
    griddep_launch_dependents();
    if (t >= T) return;
    const int h0 = static_cast<int>(gid - t * vpr) * 8;
    const int32_t *prow = pos + t * K;
    const float *wrow = w ? w + t * K : nullptr;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    bool bad = false;
    for (int k0 = 0; k0 < K; k0 += RD_LOOKAHEAD) {
        Vec8<TIn> buf[RD_LOOKAHEAD];
        bool use[RD_LOOKAHEAD];
        float wk[RD_LOOKAHEAD];
#pragma unroll
        for (int j = 0; j < RD_LOOKAHEAD; ++j) {
            use[j] = false;
            wk[j] = 1.0f;
            if (k0 + j < K) {
                const int p = __ldg(prow + k0 + j);
                use[j] = p >= 0 && p < n_rows;
                bad |= (p < -1) || (p >= n_rows);
                if (wrow) wk[j] = __ldg(wrow + k0 + j);
                if (use[j] && x_sf) wk[j] = __fmul_rn(wk[j], __ldg(x_sf + p));
                if (use[j]) buf[j] = load8<TIn>(x + static_cast<int64_t>(p) * H + h0);
            }
        }
#pragma unroll
        for (int j = 0; j < RD_LOOKAHEAD; ++j) {
            if (use[j]) {
                float f[8];
                unpack8(buf[j], f);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(wk[j], f[i]));
            }
        }
    }
    if (sf) {
        const float sv = __ldg(sf + t);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = __fmul_rn(acc[i], sv);
    }
    store8<TOut>(out + t * H + h0, acc);
    if (bad && err) atomicExch(err, kErrDeviceFlag);
}

// ---------------------------------------------------------------------------
// Persistent combine fed by bulk copies (TileOPs-Metax PR #55 section 1 "H
// tiling" and "look-ahead", done with the copy engine): a work item is one
// token and one H tile of HT elements.  Warp 0 is the producer: lane j reads
// pos[t, j] and w[t, j]; each valid slot row's H tile is fetched with one
// cp.async.bulk into a stage of a shared-memory ring (all K slots of an item
// land on the stage's mbarrier); the slot weights and the valid mask go into
// the stage header.  Warps 1..4 consume: thread i accumulates 8 hidden
// elements over the valid slots in ascending order (acc = acc + w*x, the same
// roundings as the plain definition) and stores them once.  The producer runs
// up to `stages` items ahead of the consumers.
// ---------------------------------------------------------------------------
constexpr int RB_CONSUMER_WARPS = 4;
constexpr int RB_THREADS = 32 * (1 + RB_CONSUMER_WARPS);
constexpr int RB_MAX_K = 32;
constexpr int RB_HEADER = 256;  // weights[32] + mask, padded

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

template <typename TIn>
__device__ __forceinline__ void load8_smem(const uint8_t *p, float (&f)[8]);
template <>
__device__ __forceinline__ void load8_smem<__nv_bfloat16>(const uint8_t *p, float (&f)[8]) {
    unpack8(Vec8<__nv_bfloat16>{*reinterpret_cast<const uint4 *>(p)}, f);
}
template <>
__device__ __forceinline__ void load8_smem<__half>(const uint8_t *p, float (&f)[8]) {
    unpack8(Vec8<__half>{*reinterpret_cast<const uint4 *>(p)}, f);
}
template <>
__device__ __forceinline__ void load8_smem<float>(const uint8_t *p, float (&f)[8]) {
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    unpack8(Vec8<float>{q[0], q[1]}, f);
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(RB_THREADS)
    reduce_bulk_kernel(const TIn *__restrict__ x, int64_t n_rows, const int32_t *__restrict__ pos,
                       const float *__restrict__ w, const float *__restrict__ x_sf,
                       const float *__restrict__ sf, int T, int K, int H, int HT, int stages,
                       TOut *__restrict__ out, int32_t *__restrict__ err, int pos_early) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_bytes = HT * static_cast<int>(sizeof(TIn));
    const int stage_bytes = RB_HEADER + K * row_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * stages);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (stages + s); };
    const int tiles = H / HT;
    const int64_t n_items = static_cast<int64_t>(T) * tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), RB_CONSUMER_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // Items are dealt round-robin (neighbouring CTAs read neighbouring H tiles
    // of the same rows, which keeps DRAM pages open).  The producer holds the
    // positions and weights of a group of 32/K items in its lanes (lane l has
    // slot l % K of item l / K) and loads the next group while issuing the
    // current one, so the position lookups stay off the critical path.
    if (warp == 0) {
        // ------------------------------- producer -------------------------------
        const int G = 32 / K;  // items per group
        const int my_q = lane / K, my_k = lane - (lane / K) * K;
        const bool slot_lane = lane < G * K;
        auto load_group = [&](int64_t first, int &pv, float &wv) {
            pv = -1;
            wv = 1.0f;
            const int64_t item = blockIdx.x + (first + my_q) * static_cast<int64_t>(gridDim.x);
            if (slot_lane && item < n_items) {
                const int64_t t = item / tiles;
                pv = __ldg(pos + t * K + my_k);
                if (w) wv = __ldg(w + t * K + my_k);
            }
        };
        int stage = 0;
        uint32_t phase = 0;
        long issued = 0;
        bool ok = true;
        int p_cur, p_nxt;
        float w_cur, w_nxt;
        // x, and unless the caller vouches for them the positions and
        // weights, may come from the previous kernel: wait for it first
        if (!pos_early) griddep_wait();
        load_group(0, p_cur, w_cur);
        load_group(G, p_nxt, w_nxt);
        if (pos_early) griddep_wait();
        griddep_launch_dependents();
        for (int64_t sidx = 0;; ++sidx) {
            const int64_t item = blockIdx.x + sidx * static_cast<int64_t>(gridDim.x);
            if (item >= n_items) break;
            const int q = static_cast<int>(sidx % G);
            if (q == 0 && sidx > 0) {
                p_cur = p_nxt;
                w_cur = w_nxt;
                load_group(sidx + G, p_nxt, w_nxt);
            }
            const int64_t t = item / tiles;
            const int ht = static_cast<int>(item - t * tiles);
            const bool mine = slot_lane && my_q == q;
            const bool valid = mine && p_cur >= 0 && p_cur < n_rows;
            const bool bad = mine && (p_cur < -1 || p_cur >= n_rows);
            const unsigned mask = (__ballot_sync(0xffffffffu, valid) >> (q * K)) &
                                  (K == 32 ? 0xffffffffu : ((1u << K) - 1u));
            if (__any_sync(0xffffffffu, bad) && lane == 0 && err) atomicExch(err, kErrDeviceFlag);
            int go = 1;
            if (lane == 0) go = mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, err) ? 1 : 0;
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!go) {
                ok = false;
                break;
            }
            uint8_t *st = smem + stage * stage_bytes;
            if (mine) reinterpret_cast<float *>(st)[my_k] = (valid && x_sf) ? __fmul_rn(w_cur, __ldg(x_sf + p_cur)) : w_cur;
            if (lane == 0) {
                reinterpret_cast<unsigned *>(st)[RB_MAX_K] = mask;
                mbar_arrive_expect_tx(full_bar(stage), static_cast<uint32_t>(__popc(mask) * row_bytes));
            }
            __syncwarp();
            if (valid)
                bulk_g2s(smem_u32(st + RB_HEADER + my_k * row_bytes),
                         x + static_cast<int64_t>(p_cur) * H + static_cast<int64_t>(ht) * HT,
                         static_cast<uint32_t>(row_bytes), full_bar(stage));
            ++issued;
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok && lane == 0) {
            for (long j = 1; j <= stages && j <= issued; ++j) {
                const long i = issued - j;
                rb_wait_drain(full_bar(static_cast<int>(i % stages)), static_cast<uint32_t>((i / stages) & 1));
            }
        }
    } else {
        // ------------------------------- consumers ------------------------------
        griddep_wait();  // out may still be read by the previous kernel
        griddep_launch_dependents();
        const int ct = threadIdx.x - 32;  // 0 .. 127
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
            const int64_t t = item / tiles;
            const int ht = static_cast<int>(item - t * tiles);
            int go = 1;
            if (lane == 0) go = mbar_wait_bounded(full_bar(stage), phase, abort_flag, err) ? 1 : 0;
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!go) break;
            const uint8_t *st = smem + stage * stage_bytes;
            const unsigned mask = reinterpret_cast<const unsigned *>(st)[RB_MAX_K];
            for (int v = ct; v < HT / 8; v += 32 * RB_CONSUMER_WARPS) {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                for (int k = 0; k < K; ++k) {
                    if ((mask >> k) & 1u) {
                        const float wk = reinterpret_cast<const float *>(st)[k];
                        float f[8];
                        load8_smem<TIn>(st + RB_HEADER + k * row_bytes + v * 8 * static_cast<int>(sizeof(TIn)), f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(wk, f[i]));
                    }
                }
                if (sf) {
                    const float sv = __ldg(sf + t);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = __fmul_rn(acc[i], sv);
                }
                store8<TOut>(out + t * H + static_cast<int64_t>(ht) * HT + v * 8, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(stage));
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// moe_wait_flag: lane 0 polls the flag with system-scope loads (a flag in
// pinned host memory written by the host is seen), sleeping between polls;
// the wait is bounded by the global timer and reports a timeout in *err.
// Launched without programmatic dependent launch: work after it on the
// stream starts only once it has returned.
__global__ void __launch_bounds__(32)
    wait_flag_kernel(const int32_t *flag, int32_t expected, unsigned long long timeout_ns, int32_t *err) {
    if (threadIdx.x != 0) return;
    const unsigned long long start = global_timer_ns();
    for (;;) {
        int32_t v;
        asm volatile("ld.relaxed.sys.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v >= expected) break;
        if (global_timer_ns() - start > timeout_ns) {
            atomicExch(err, kErrTimeout);
            break;
        }
        __nanosleep(1000);
    }
    // order what the flag's writer stored before the flag ahead of later work
    __threadfence_system();
}

template <typename TIn, typename TOut>
cudaError_t launch_reduce_bulk(const void *x, int64_t n_rows, const int32_t *pos, const float *w,
                               const float *x_sf, const float *sf, int64_t T, int64_t K, int64_t H,
                               void *out, int32_t *err, cudaStream_t stream, bool pos_early) {
    // H tile: the largest of 1024 / 512 / 256 that divides H with a slot row <= 2 KB
    int HT = 256;
    for (int cand : {1024, 512}) {
        if (H % cand == 0 && cand * static_cast<int>(sizeof(TIn)) <= 2048) {
            HT = cand;
            break;
        }
    }
    // about 64 KB of ring per CTA, three CTAs per SM (measured best among
    // 1-2 KB tiles, 2-6 stages and 2-8 CTAs per SM at 512 and 4096 tokens)
    const int stage_bytes = RB_HEADER + static_cast<int>(K) * HT * static_cast<int>(sizeof(TIn));
    int stages = (68 * 1024) / stage_bytes;
    stages = stages < 2 ? 2 : (stages > 6 ? 6 : stages);
    const size_t smem = static_cast<size_t>(stages) * stage_bytes + 16 * stages + 16;
    auto kern = reduce_bulk_kernel<TIn, TOut>;
    static std::atomic<size_t> attr_bytes[64];  // zero-initialised; several host threads may launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (smem > 48 * 1024 && (dev < 0 || dev >= 64 || attr_bytes[dev] < smem)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_bytes[dev] = smem;
    }
    const int per_sm = static_cast<int>((200 * 1024) / smem) < 1 ? 1 : static_cast<int>((200 * 1024) / smem);
    const int64_t n_items = T * (H / HT);
    int64_t grid = static_cast<int64_t>(device_sm_count()) * (per_sm > 3 ? 3 : per_sm);
    if (grid > n_items) grid = n_items;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(RB_THREADS), smem, stream,
                      static_cast<const TIn *>(x), n_rows, pos, w, x_sf, sf, static_cast<int>(T),
                      static_cast<int>(K), static_cast<int>(H), HT, stages,
                      static_cast<TOut *>(out), err, pos_early ? 1 : 0);
}

template <typename TIn, typename TOut>
cudaError_t launch_reduce_typed(const void *x, int64_t n_rows, const int32_t *pos, const float *w,
                                const float *x_sf, const float *sf, int64_t T, int64_t K,
                                int64_t H, void *out, int32_t *err, cudaStream_t stream, bool pos_early) {
    if (K <= RB_MAX_K)
        return launch_reduce_bulk<TIn, TOut>(x, n_rows, pos, w, x_sf, sf, T, K, H, out, err, stream,
                                             pos_early);
    const int64_t threads = T * (H / 8);
    const int64_t blocks = (threads + RD_THREADS - 1) / RD_THREADS;
    return launch_pdl(reduce_fused_kernel<TIn, TOut>, dim3(static_cast<unsigned>(blocks)),
                      dim3(RD_THREADS), 0, stream, static_cast<const TIn *>(x), n_rows, pos, w,
                      x_sf, sf, T, static_cast<int>(K), static_cast<int>(H),
                      static_cast<TOut *>(out), err);
}

template <typename TIn>
cudaError_t launch_reduce_in(const void *x, int64_t n_rows, const int32_t *pos, const float *w,
                             const float *x_sf, const float *sf, int64_t T, int64_t K, int64_t H,
                             int out_dtype, void *out, int32_t *err, cudaStream_t stream, bool pe) {
    switch (out_dtype) {
        case kF16: return launch_reduce_typed<TIn, __half>(x, n_rows, pos, w, x_sf, sf, T, K, H, out, err, stream, pe);
        case kBF16: return launch_reduce_typed<TIn, __nv_bfloat16>(x, n_rows, pos, w, x_sf, sf, T, K, H, out, err, stream, pe);
        case kF32: return launch_reduce_typed<TIn, float>(x, n_rows, pos, w, x_sf, sf, T, K, H, out, err, stream, pe);
        case kE4M3: return launch_reduce_typed<TIn, __nv_fp8_e4m3>(x, n_rows, pos, w, x_sf, sf, T, K, H, out, err, stream, pe);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gather_rows(const void *x, const int32_t *sorted_token_idx, int64_t n_rows,
                               int64_t d_h, int elem_bytes, void *a_out, cudaStream_t stream) {
    if (n_rows <= 0) return cudaSuccess;
    const int nvec = static_cast<int>(d_h * elem_bytes / 16);
    const int64_t blocks = (n_rows + GA_WARPS - 1) / GA_WARPS;
    return launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(GA_WARPS * 32), 0,
                      stream, static_cast<const uint4 *>(x), sorted_token_idx, n_rows, nvec,
                      static_cast<uint4 *>(a_out));
}

cudaError_t launch_scatter_rows(const void *x, const int32_t *token_topk_to_pos, int64_t T, int64_t k,
                                int64_t n_rows, int64_t d_h, int elem_bytes, void *a_out, int32_t *err,
                                cudaStream_t stream) {
    if (T <= 0 || n_rows <= 0) return cudaSuccess;
    if (k <= 0 || k > 32) return cudaErrorInvalidValue;
    const int64_t row_bytes = d_h * elem_bytes;
    const int64_t buf_bytes = (row_bytes + 127) / 128 * 128;
    int64_t wpc = SB_SMEM_BUDGET / (2 * buf_bytes + 16);
    if (wpc > SB_MAX_WARPS) wpc = SB_MAX_WARPS;
    if (wpc >= 1 && row_bytes < (1 << 20)) {
        // bulk form: resident CTAs only (a persistent grid of token streams)
        static std::atomic<bool> attr_done[64];  // zero-initialised; several host threads may launch
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
        if (dev < 0 || dev >= 64 || !attr_done[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(scatter_rows_bulk_kernel,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       SB_SMEM_BUDGET + SB_MAX_WARPS * 16);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_done[dev] = true;
        }
        const int64_t smem = wpc * (2 * buf_bytes + 16);
        int smem_sm = 0, reserved = 0;
        if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
            return cudaErrorInvalidDevice;
        int64_t per_sm = smem_sm / (smem + reserved);
        const int64_t by_threads = 2048 / (wpc * 32);
        if (per_sm > by_threads) per_sm = by_threads;
        if (per_sm >= 1) {
            const int64_t want = (T + wpc - 1) / wpc;
            const int64_t cap = static_cast<int64_t>(device_sm_count()) * per_sm;
            const int64_t blocks = want < cap ? want : cap;
            return launch_pdl(scatter_rows_bulk_kernel, dim3(static_cast<unsigned>(blocks)),
                              dim3(static_cast<unsigned>(wpc * 32)), static_cast<size_t>(smem), stream,
                              static_cast<const uint8_t *>(x), token_topk_to_pos, T, static_cast<int>(k), n_rows,
                              static_cast<uint32_t>(row_bytes), static_cast<uint32_t>(buf_bytes),
                              static_cast<uint8_t *>(a_out), err);
        }
    }
    const int nvec = static_cast<int>(d_h * elem_bytes / 16);
    const int64_t blocks = (T + GA_WARPS - 1) / GA_WARPS;
    return launch_pdl(scatter_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(GA_WARPS * 32), 0, stream,
                      static_cast<const uint4 *>(x), token_topk_to_pos, T, static_cast<int>(k), n_rows, nvec,
                      static_cast<uint4 *>(a_out));
}

cudaError_t launch_copy(const void *src, void *dst, int64_t bytes, cudaStream_t stream) {
    if (bytes <= 0) return cudaSuccess;
    const int64_t nvec = bytes / 16;
    // enough threads for one vector each up to 152 x 8 CTAs, then 4 per pass
    const int64_t want = (nvec + CP_THREADS - 1) / CP_THREADS;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    const int blocks = static_cast<int>(want < cap ? want : cap);
    return launch_pdl(copy_kernel, dim3(static_cast<unsigned>(blocks)), dim3(CP_THREADS), 0, stream,
                      static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), nvec);
}

cudaError_t launch_wait_flag(const int32_t *flag, int32_t expected, int64_t timeout_ns, int32_t *err,
                             cudaStream_t stream) {
    wait_flag_kernel<<<1, 32, 0, stream>>>(flag, expected, static_cast<unsigned long long>(timeout_ns), err);
    return cudaGetLastError();
}

cudaError_t launch_reduce_fused(const void *x, int64_t n_rows, const int32_t *pos,
                                const float *w, const float *x_sf, const float *sf, int64_t T,
                                int64_t K, int64_t H, int in_dtype, int out_dtype, void *out,
                                int32_t *err, cudaStream_t stream, bool pos_early) {
    if (T <= 0) return cudaSuccess;
    const bool pe = pos_early;
    switch (in_dtype) {
        case kF16: return launch_reduce_in<__half>(x, n_rows, pos, w, x_sf, sf, T, K, H, out_dtype, out, err, stream, pe);
        case kBF16: return launch_reduce_in<__nv_bfloat16>(x, n_rows, pos, w, x_sf, sf, T, K, H, out_dtype, out, err, stream, pe);
        case kF32: return launch_reduce_in<float>(x, n_rows, pos, w, x_sf, sf, T, K, H, out_dtype, out, err, stream, pe);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe

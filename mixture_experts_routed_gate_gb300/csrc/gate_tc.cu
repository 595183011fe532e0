// gate_tc.cu -- gate logits on the tensor cores for many tokens, with the
// routing kept exactly what the fixed summation order gives.
//
// The routing (top-k ids, their order, the tables built from them) is defined
// by logits summed in one fixed order (8-element chunks, chunk c by warp lane
// c mod 32 in ascending index with fmaf, the 32 partials combined by the xor
// butterfly 16, 8, 4, 2, 1, then + bias).  A tensor-core product sums in
// another order, so its logits can differ in the last bits and could swap two
// experts whose logits nearly tie.  This path therefore:
//
//   1. gate_tc_kernel: logits~ = x W_g^T on the tensor cores (tcgen05, fp32
//      accumulation, operands by TMA through two rings: token rows, read
//      once from DRAM, in the deeper one; gate rows, re-read from L2 by
//      every token tile, in the other), K split over S CTAs per output tile
//      (partials [S, T, E], written by tensor stores from the idle ring);
//      the otherwise idle epilogue warps also compute |w_e|_2 for every gate
//      row and, from the token tiles in shared memory, each split's share of
//      |x_t|^2.
//   2. gate_select_kernel, one warp per token: sums the partials in a fixed
//      order, bounds |logit~ - logit| <= delta(t, e) from |x_t|_2 |w_e|_2
//      (Cauchy-Schwarz on sum |x_j w_j|) and the rounding depth of both
//      orders, and keeps as candidates every expert whose upper bound reaches
//      the k-th largest lower bound.  An expert outside that set has a logit
//      strictly below k others, so it cannot be selected.  Every candidate's
//      logit is then recomputed in the fixed order (the same bits as the
//      CUDA-core gate), and the top-k is chosen among the candidates by
//      (logit desc, id asc); the k-th lower bound and the top-k are integer
//      warp reductions on order-preserving keys of the floats.  Weights: softmax at the selected experts, the
//      denominator over the fixed-order logits of the candidates and the
//      tensor-core logits of the others (their terms are below the k-th
//      largest and within delta of exact).
//
// Error model behind delta (stated, not measured): one tcgen05 K=16 MMA step
// returns the fp32 accumulator within 18 * 2^-23 * max(|acc_in|, |products|)
// of the exact sum (17 addends, each aligned to the largest and truncated to
// fp32 precision, plus the final rounding; products of two 16-bit values are
// exact in fp32); a split of G such steps is then within 18 G 2^-23 of its
// own sum |x_j w_j|, the fixed order within (d_h/32 + 5) 2^-24 of it, and the
// S partials and the bias add S + 2 more roundings.  delta doubles that sum
// of bounds and adds 2^-22 |logit~| for the final bias rounding on both sides.
// If any value is not finite every expert becomes a candidate.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int GT_BM = 128;       // tokens per tile (MMA M)
constexpr int GT_BN = 256;       // experts per tile (MMA N)
constexpr int GT_BK = 64;        // 64 x 2 B = one 128-byte swizzle row
// Two rings: token rows come from DRAM (read once), gate rows from L2 (every
// token tile reads them), so the token ring is the deeper one.
constexpr int GT_XS = 6;         // token-row stages (16 KB each)
constexpr int GT_WS = 3;         // gate-row stages (32 KB each)
constexpr int GT_THREADS = 192;  // warp 0 TMA (lane 0 token rows, lane 1 gate rows), warp 1 MMA, warps 2-5 epilogue
constexpr int GT_A_BYTES = GT_BM * GT_BK * 2;
constexpr int GT_B_BYTES = GT_BN * GT_BK * 2;
constexpr int GT_SMEM = 1024 + GT_XS * GT_A_BYTES + GT_WS * GT_B_BYTES + 256;
static_assert(GT_SMEM <= 227 * 1024, "shared memory per CTA");
constexpr int GT_MAX_SPLITS = 8;
constexpr int SEL_WARPS = 4;     // warps (tokens) of a select CTA
constexpr int SEL_G = 3;         // candidates recomputed together by a warp
constexpr int SEL_U = 4;         // chunks per lane whose loads are in flight together

struct GateTcParams {
    float *part;           // [S, T, E] fp32 partial logits (no bias)
    int tma_store;         // 1: the partials leave through tm_p (E % 4 == 0)
    float *wnorm;          // [E] |w_e|_2
    float *xss;            // [S, T] sum of x_t^2 over each split's columns
    const uint8_t *wg;     // gate weight [E, d_h], 16-bit elements
    int T, E, d_h;
    int nk;                // 64-wide K steps in d_h
    int ks;                // K steps per split
    int *err;
};

// Sum of squares of one row of d_h 16-bit values, by a warp (every lane
// gets the total).  Eight 16-byte loads in flight per lane, one partial sum
// per load (any fp32 order: the sum only enters the error bound).
template <int DT>
__device__ __forceinline__ float row_sumsq(const uint8_t *row_bytes, int d_h, int lane) {
    const uint4 *row = reinterpret_cast<const uint4 *>(row_bytes);
    const int chunks = d_h / 8;
    float ssu[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) ssu[u] = 0.0f;
    for (int cb = lane; cb < chunks; cb += 32 * 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (cb + 32 * u < chunks) v[u] = __ldg(row + cb + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (cb + 32 * u < chunks) {
                const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = unpack2<DT>(w4[q]);
                    ssu[u] = fmaf(f.x, f.x, ssu[u]);
                    ssu[u] = fmaf(f.y, f.y, ssu[u]);
                }
            }
        }
    }
    float ss = ((ssu[0] + ssu[1]) + (ssu[2] + ssu[3])) + ((ssu[4] + ssu[5]) + (ssu[6] + ssu[7]));
#pragma unroll
    for (int sh = 16; sh >= 1; sh >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, sh);
    return ss;
}

// shared -> global tensor store of one box (3-D map), in the CTA's bulk group
__device__ __forceinline__ void tma_store_3d(const void *desc, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(desc)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

template <int DT>
__global__ void __launch_bounds__(GT_THREADS, 1)
    gate_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                   const __grid_constant__ CUtensorMap tm_p, const GateTcParams p) {
    constexpr uint32_t IDESC = idesc_f16(DT == kBF16, GT_BM, GT_BN);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + GT_XS * GT_A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + GT_WS * GT_B_BYTES);
    constexpr int NBARS = 2 * GT_XS + 2 * GT_WS + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    static_assert(NBARS * 8 + 8 <= 256, "barrier area");
    const uint32_t bar0 = smem_u32(bars);
    auto xfull_bar = [&](int s) { return bar0 + 8u * s; };
    auto xempty_bar = [&](int s) { return bar0 + 8u * (GT_XS + s); };
    auto wfull_bar = [&](int s) { return bar0 + 8u * (2 * GT_XS + s); };
    auto wempty_bar = [&](int s) { return bar0 + 8u * (2 * GT_XS + GT_WS + s); };
    const uint32_t acc_bar = bar0 + 8u * (2 * GT_XS + 2 * GT_WS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * GT_BM, n0 = blockIdx.y * GT_BN, split = blockIdx.z;
    const int kb0 = split * p.ks;
    const int kb1 = min(p.nk, kb0 + p.ks);

    if (threadIdx.x == 0) {
        for (int s = 0; s < GT_XS; ++s) {
            mbar_init(xfull_bar(s), 1);
            // a token stage is free once its MMAs completed (commit) and
            // every epilogue warp has read its token rows' squares from it
            mbar_init(xempty_bar(s), 1 + 4);
        }
        for (int s = 0; s < GT_WS; ++s) {
            mbar_init(wfull_bar(s), 1);
            mbar_init(wempty_bar(s), 1);  // its MMAs completed
        }
        mbar_init(acc_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), GT_BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();  // x may come from the previous kernel
    griddep_launch_dependents();

    if (warp == 0) {
        if (lane < 2) {
            // ------------------------------ TMA producers -----------------------------
            // lane 0: the token rows (ring of GT_XS); lane 1: the gate rows (GT_WS)
            const bool xr = lane == 0;
            const int nst = xr ? GT_XS : GT_WS;
            const uint32_t bytes = xr ? GT_A_BYTES : GT_B_BYTES;
            int stage = 0;
            uint32_t phase = 0;
            long issued = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_bounded(xr ? xempty_bar(stage) : wempty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = xr ? xfull_bar(stage) : wfull_bar(stage);
                mbar_arrive_expect_tx(fb, bytes);
                // rows past T or E read as zero
                if (xr)
                    tma_load_2d(smem_u32(sA + stage * GT_A_BYTES), &tm_x, fb, kb * GT_BK, m0);
                else
                    tma_load_2d(smem_u32(sB + stage * GT_B_BYTES), &tm_w, fb, kb * GT_BK, n0);
                ++issued;
                if (++stage == nst) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                // let the copies in flight land before shared memory goes away
                for (long j = 1; j <= nst && j <= issued; ++j) {
                    const long i = issued - j;
                    const int st = static_cast<int>(i % nst);
                    const uint32_t bar = xr ? xfull_bar(st) : wfull_bar(st);
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_try_wait(bar, static_cast<uint32_t>((i / nst) & 1)))
                        if (global_timer_ns() - t0 > kWaitTimeoutNs) break;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------- MMA issuer --------------------------------
            int xs = 0, ws = 0;
            uint32_t xphase = 0, wphase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_bounded(xfull_bar(xs), xphase, abort_flag, p.err) ||
                    !mbar_wait_bounded(wfull_bar(ws), wphase, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t a_desc = smem_desc_sw128(smem_u32(sA + xs * GT_A_BYTES));
                const uint64_t b_desc = smem_desc_sw128(smem_u32(sB + ws * GT_B_BYTES));
#pragma unroll
                for (int k = 0; k < GT_BK / 16; ++k)
                    tc_mma_f16(tmem_base, a_desc + 2u * k, b_desc + 2u * k, IDESC,
                               (kb > kb0 || k > 0) ? 1u : 0u);
                tc_commit(xempty_bar(xs));
                tc_commit(wempty_bar(ws));
                if (++xs == GT_XS) {
                    xs = 0;
                    xphase ^= 1u;
                }
                if (++ws == GT_WS) {
                    ws = 0;
                    wphase ^= 1u;
                }
            }
            // the accumulator (or, after an abort, the last MMAs) is complete
            tc_commit(acc_bar);
            if (!ok) {
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(acc_bar, 0))
                    if (global_timer_ns() - t0 > kWaitTimeoutNs) break;
            }
        }
    } else {
        // -------------------------------- epilogue --------------------------------
        // while the main loop runs: the sum of squares of this thread's token
        // row over the split's columns, read from each stage's A tile (the
        // row's 128 bytes; the swizzle only permutes 16-byte chunks inside
        // them) before the stage is released.  This read releases the stage,
        // so it paces the main loop: thread `row` reads its chunks starting
        // at chunk row % 8, so the eight threads of a 16-byte access phase
        // hit eight different bank groups (reading chunk c in every row put
        // all of them on the same four banks), and eight partial sums keep
        // the chain short (the sum only enters the error bound, whose slack
        // covers any fp32 summation order).
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int t = m0 + row;
        {
            int stage = 0;
            uint32_t phase = 0;
            float ssc[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) ssc[c] = 0.0f;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                int go = 1;
                if (lane == 0) go = mbar_wait_bounded(xfull_bar(stage), phase, abort_flag, p.err) ? 1 : 0;
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
                const uint4 *r = reinterpret_cast<const uint4 *>(sA + stage * GT_A_BYTES + row * 128);
                uint4 v[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) v[c] = r[(c + row) & 7];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 f = unpack2<DT>(w4[h]);
                        ssc[c] = fmaf(f.x, f.x, ssc[c]);
                        ssc[c] = fmaf(f.y, f.y, ssc[c]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(xempty_bar(stage));
                if (++stage == GT_XS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            const float ss = ((ssc[0] + ssc[1]) + (ssc[2] + ssc[3])) + ((ssc[4] + ssc[5]) + (ssc[6] + ssc[7]));
            if (ok && blockIdx.y == 0 && t < p.T) p.xss[static_cast<int64_t>(split) * p.T + t] = ss;
        }
        // |w_e|_2 of a share of the gate rows (all CTAs together cover every
        // row once), while the last MMAs run
        {
            const int n_cta = gridDim.x * gridDim.y * gridDim.z;
            const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
            const int gw = cta * 4 + (warp - 2);
            for (int e = gw; e < p.E; e += n_cta * 4) {
                const float ss = row_sumsq<DT>(p.wg + static_cast<int64_t>(e) * p.d_h * 2, p.d_h, lane);
                if (lane == 0) p.wnorm[e] = sqrtf(ss);
            }
        }
        // then the partial logits of this tile and split: thread = token row
        int ready = 1;
        if (lane == 0) ready = mbar_wait_bounded(acc_bar, 0, abort_flag, p.err) ? 1 : 0;
        ready = __shfl_sync(0xffffffffu, ready, 0);
        // every epilogue warp is past its reads of the token stages before
        // the ring is reused for the staged tile
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (ready) {
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            if (p.tma_store) {
                // the tile in the idle ring as GT_BN / 32 boxes of 128 token rows x 32
                // experts (128-byte rows, 16-byte chunks swizzled by row % 8, as the
                // store's tensor map reads them; eight rows of a warp's store fill
                // all banks once)
#pragma unroll 1
                for (int b = 0; b < GT_BN / 32; ++b) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(t_row + b * 32, r0);
                    tmem_ld16(t_row + b * 32 + 16, r1);
                    tmem_ld_wait();
                    uint8_t *rowp = smem + b * (GT_BM * 128) + row * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        *reinterpret_cast<uint4 *>(rowp + ((c ^ (row & 7)) * 16)) =
                            make_uint4(r0[4 * c], r0[4 * c + 1], r0[4 * c + 2], r0[4 * c + 3]);
                        *reinterpret_cast<uint4 *>(rowp + (((c + 4) ^ (row & 7)) * 16)) =
                            make_uint4(r1[4 * c], r1[4 * c + 1], r1[4 * c + 2], r1[4 * c + 3]);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            } else {
                float *out = p.part + (static_cast<int64_t>(split) * p.T + (t < p.T ? t : 0)) * p.E;
#pragma unroll 1
                for (int c = 0; c < GT_BN / 16; ++c) {
                    uint32_t r[16];
                    tmem_ld16(t_row + c * 16, r);
                    tmem_ld_wait();
                    const int e0 = n0 + c * 16;
                    if (t < p.T && e0 < p.E) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (e0 + i < p.E) out[e0 + i] = __uint_as_float(r[i]);
                    }
                }
            }
        }
        if (p.tma_store) {
            asm volatile("bar.sync 1, 128;" ::: "memory");  // every row staged
            if (warp == 2 && lane == 0 && ready) {
                // rows past T (per split) and experts past E are clipped by the map
                for (int b = 0; b < GT_BN / 32; ++b)
                    if (n0 + 32 * b < p.E) tma_store_3d(&tm_p, smem_u32(smem + b * (GT_BM * 128)), n0 + 32 * b, m0, split);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, GT_BN);
    }
}

// Order-preserving key of a float that is not NaN (-0 taken as +0): a > b
// as floats exactly when key(a) > key(b); 0 is below every key.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One chunk of NG candidates' chains: the 8 elements in ascending order, each
// a single-rounding fmaf on the exactly widened 16-bit values (the same bits
// as the mixed-precision FMA of the CUDA-core gate); x is widened once for all
// NG chains.
template <int DT, int NG>
__device__ __forceinline__ void select_chunk(const uint4 &xv, const uint4 *wv, float *acc) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 xf = unpack2<DT>(xw[q]);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const uint32_t w = q == 0 ? wv[g].x : q == 1 ? wv[g].y : q == 2 ? wv[g].z : wv[g].w;
            const float2 wf = unpack2<DT>(w);
            acc[g] = fmaf(xf.x, wf.x, acc[g]);
            acc[g] = fmaf(xf.y, wf.y, acc[g]);
        }
    }
}

// Lane `lane`'s chains of NG candidates (rows off[g] / chunks of the gate
// weight): chunks c = lane, lane + 32, ... in ascending order, SEL_U chunks'
// loads in flight.
template <int DT, int NG>
__device__ __forceinline__ void select_chains(const uint4 *__restrict__ xrow, const uint4 *__restrict__ wbase,
                                              const int *off, int chunks, int lane, float *acc) {
    int c = lane;
    for (; c + 32 * (SEL_U - 1) < chunks; c += 32 * SEL_U) {
        uint4 xv[SEL_U], wv[SEL_U][NG];
#pragma unroll
        for (int u = 0; u < SEL_U; ++u) {
            xv[u] = __ldg(xrow + c + 32 * u);
#pragma unroll
            for (int g = 0; g < NG; ++g) wv[u][g] = __ldg(wbase + off[g] + c + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < SEL_U; ++u) select_chunk<DT, NG>(xv[u], wv[u], acc);
    }
    for (; c < chunks; c += 32) {
        uint4 wv[NG];
        const uint4 xv = __ldg(xrow + c);
#pragma unroll
        for (int g = 0; g < NG; ++g) wv[g] = __ldg(wbase + off[g] + c);
        select_chunk<DT, NG>(xv, wv, acc);
    }
}

// select_chains with NG = ng (1 <= ng <= NG), so a short last group runs
// only its own chains.
template <int DT, int NG>
__device__ __forceinline__ void select_group(int ng, const uint4 *xrow, const uint4 *wbase, const int *off,
                                             int chunks, int lane, float *acc) {
    if constexpr (NG > 1) {
        if (ng < NG) {
            select_group<DT, NG - 1>(ng, xrow, wbase, off, chunks, lane, acc);
            return;
        }
    }
    select_chains<DT, NG>(xrow, wbase, off, chunks, lane, acc);
}

// One warp per token, SEL_WARPS tokens per CTA.  The warp sums the partials
// in split order, forms the bounds and the candidate list, recomputes every
// candidate in the fixed order (SEL_G candidates at a time: lane L runs one
// accumulator chain per candidate over its chunks c = L, L + 32, ... in
// ascending order, the chains interleaved, SEL_U chunks' loads in flight),
// then selects the top-k and forms the weights.  Shared memory per warp: per
// expert its logit (the tensor-core value, replaced by the fixed-order value
// for candidates), the candidate ids and their fixed-order logits.
template <int DT, int SLOTS>
__global__ void __launch_bounds__(SEL_WARPS * 32)
    gate_select_kernel(const uint8_t *__restrict__ x, const uint8_t *__restrict__ wg,
                       const float *__restrict__ bias, const float *__restrict__ part,
                       const float *__restrict__ wnorm, const float *__restrict__ xss, int T, int E,
                       int d_h, int S, int k, float coef, float *__restrict__ logits,
                       int32_t *__restrict__ topk_idx, float *__restrict__ topk_w) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *val = reinterpret_cast<float *>(sel_smem) + static_cast<int64_t>(warp) * 3 * E;
    int *cand_id = reinterpret_cast<int *>(val + E);
    float *cand_val = reinterpret_cast<float *>(cand_id + E);
    const int t = blockIdx.x * SEL_WARPS + warp;
    const int chunks = d_h / 8;
    griddep_wait();  // partials and norms come from gate_tc_kernel
    griddep_launch_dependents();
    if (t >= T) return;

    int n = 0;  // candidates (warp-uniform)
    {
        float xv[8];
#pragma unroll
        for (int sp = 0; sp < 8; ++sp) xv[sp] = sp < S ? xss[static_cast<int64_t>(sp) * T + t] : 0.0f;
        float xsum = xv[0];
#pragma unroll
        for (int sp = 1; sp < 8; ++sp)
            if (sp < S) xsum = xsum + xv[sp];
        const float xn = sqrtf(xsum);
        // tensor-core logits (partials summed in split order, then + bias) and bounds
        float lo[SLOTS], hi[SLOTS];
        bool bad = !isfinite(xn);
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int e = s * 32 + lane;
            lo[s] = -INFINITY;
            hi[s] = -INFINITY;
            if (e < E) {
                float pv[8];
#pragma unroll
                for (int sp = 0; sp < 8; ++sp)
                    pv[sp] = sp < S ? part[(static_cast<int64_t>(sp) * T + t) * E + e] : 0.0f;
                float l = pv[0];
#pragma unroll
                for (int sp = 1; sp < 8; ++sp)
                    if (sp < S) l = l + pv[sp];
                const float b = bias ? bias[e] : 0.0f;
                if (bias) l = l + b;
                const float d = coef * fmaf(xn, wnorm[e], fabsf(b)) + 0x1.0p-22f * fabsf(l) + 1e-30f;
                val[e] = l;
                lo[s] = l - d;
                hi[s] = l + d;
                bad |= !isfinite(l) || !isfinite(d);
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        // theta = k-th largest lower bound: k rounds of a warp max (one
        // integer reduction) over order-preserving keys; each round clears one
        // holder of the maximum
        float theta = -INFINITY;
        if (!bad) {
            uint32_t key[SLOTS];
#pragma unroll
            for (int s = 0; s < SLOTS; ++s) key[s] = s * 32 + lane < E ? order_key(lo[s]) : 0u;
            uint32_t kth = 0u;
            for (int j = 0; j < k; ++j) {
                uint32_t m = 0u;
#pragma unroll
                for (int s = 0; s < SLOTS; ++s) m = max(m, key[s]);
                kth = __reduce_max_sync(0xffffffffu, m);
                const unsigned holders = __ballot_sync(0xffffffffu, m == kth);
                if (lane == __ffs(holders) - 1) {
                    bool done = false;
#pragma unroll
                    for (int s = 0; s < SLOTS; ++s) {
                        if (!done && key[s] == kth) {
                            key[s] = 0u;
                            done = true;
                        }
                    }
                }
            }
            if (kth != 0u) theta = key_value(kth);
        }
        // candidates, in ascending expert id
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int e = s * 32 + lane;
            const bool c = e < E && (bad || hi[s] >= theta);
            const unsigned m = __ballot_sync(0xffffffffu, c);
            if (c) cand_id[n + __popc(m & ((1u << lane) - 1u))] = e;
            n += __popc(m);
        }
    }
    __syncwarp();

    // fixed-order logits of the candidates, SEL_G at a time
    const uint4 *xrow = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t) * d_h * 2);
    const uint4 *wbase = reinterpret_cast<const uint4 *>(wg);
    for (int i0 = 0; i0 < n; i0 += SEL_G) {
        const int ng = min(SEL_G, n - i0);
        int off[SEL_G];
        float acc[SEL_G];
#pragma unroll
        for (int g = 0; g < SEL_G; ++g) {
            off[g] = cand_id[i0 + (g < ng ? g : 0)] * chunks;
            acc[g] = 0.0f;
        }
        select_group<DT, SEL_G>(ng, xrow, wbase, off, chunks, lane, acc);
#pragma unroll
        for (int g = 0; g < SEL_G; ++g) {
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) acc[g] = acc[g] + __shfl_xor_sync(0xffffffffu, acc[g], sh);
            if (g < ng) {
                const int e = off[g] / chunks;
                if (bias) acc[g] = acc[g] + bias[e];
                if (lane == 0) {
                    cand_val[i0 + g] = acc[g];
                    val[e] = acc[g];
                }
            }
        }
    }
    __syncwarp();

    // top-k among the candidates by (logit desc, id asc); lane j keeps slot j.
    // At most 32 candidates, none NaN: one per lane, each round a warp max of
    // the keys and a warp min of the ids holding it.  Otherwise a scan.
    float top = 0.0f, my_v = 0.0f;
    int my_e = 0;
    bool one_each = n <= 32;
    float cv = 0.0f;
    int ce = 0;
    if (one_each) {
        if (lane < n) {
            cv = cand_val[lane];
            ce = cand_id[lane];
        }
        one_each = !__any_sync(0xffffffffu, lane < n && isnan(cv));
    }
    if (one_each) {
        uint32_t key = lane < n ? order_key(cv) : 0u;
        for (int j = 0; j < k; ++j) {
            const uint32_t m = __reduce_max_sync(0xffffffffu, key);
            const uint32_t be =
                __reduce_min_sync(0xffffffffu, key == m && key != 0u ? static_cast<uint32_t>(ce) : 0xffffffffu);
            if (key == m && static_cast<uint32_t>(ce) == be) key = 0u;
            const float bv = key_value(m);
            if (j == 0) top = bv;
            if (j == lane) {
                my_v = bv;
                my_e = static_cast<int>(be);
            }
        }
    } else {
        unsigned taken = 0;  // bit i: candidate lane + 32 i already selected
        for (int j = 0; j < k; ++j) {
            float best = -INFINITY;
            int best_e = 0x7fffffff, best_i = -1;
            for (int i = lane, b = 0; i < n; i += 32, ++b) {
                if (taken & (1u << b)) continue;
                const float v = cand_val[i];
                const int e = cand_id[i];
                if (best_i < 0 || v > best || (v == best && e < best_e)) {
                    best = v;
                    best_e = e;
                    best_i = i;
                }
            }
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) {
                const float ob = __shfl_xor_sync(0xffffffffu, best, sh);
                const int oe = __shfl_xor_sync(0xffffffffu, best_e, sh);
                const int oi = __shfl_xor_sync(0xffffffffu, best_i, sh);
                if (oi >= 0 && (best_i < 0 || ob > best || (ob == best && oe < best_e))) {
                    best = ob;
                    best_e = oe;
                    best_i = oi;
                }
            }
            if (best_i >= 0 && (best_i & 31) == lane) taken |= 1u << (best_i >> 5);
            if (j == 0) top = best;
            if (j == lane) {
                my_v = best;
                my_e = best_e;
            }
        }
    }
    // softmax denominator over every expert (per lane in slot order, then the
    // butterfly), the logits row written once
    float sum = 0.0f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int e = s * 32 + lane;
        if (e < E) {
            const float v = val[e];
            sum += expf(v - top);
            logits[static_cast<int64_t>(t) * E + e] = v;
        }
    }
#pragma unroll
    for (int sh = 16; sh >= 1; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
    if (lane < k) {
        topk_idx[static_cast<int64_t>(t) * k + lane] = my_e;
        topk_w[static_cast<int64_t>(t) * k + lane] = expf(my_v - top) / sum;
    }
}

size_t select_smem_bytes(int64_t d_h, int64_t E) {
    (void)d_h;
    return static_cast<size_t>(SEL_WARPS * E * 12);
}

int splits_for(int64_t T, int64_t E) {
    const int64_t tiles = ((T + GT_BM - 1) / GT_BM) * ((E + GT_BN - 1) / GT_BN);
    int64_t s = 128 / (tiles > 0 ? tiles : 1);
    return static_cast<int>(s < 1 ? 1 : (s > GT_MAX_SPLITS ? GT_MAX_SPLITS : s));
}

template <int DT>
cudaError_t launch_typed(const void *x, const void *wg, const float *bias, int64_t T, int64_t d_h,
                         int64_t E, int64_t k, float *logits, float *part, float *wnorm, float *xss,
                         int32_t *topk_idx, float *topk_w, int32_t *err, cudaStream_t stream) {
    const int nk = static_cast<int>(d_h / GT_BK);
    int S = splits_for(T, E);
    if (S > nk) S = nk;
    const int ks = (nk + S - 1) / S;
    S = (nk + ks - 1) / ks;  // every split non-empty
    CUtensorMap tm_x, tm_w;
    const int cu_dt = DT == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t dx[2] = {static_cast<uint64_t>(d_h), static_cast<uint64_t>(T)};
    const uint64_t dw[2] = {static_cast<uint64_t>(d_h), static_cast<uint64_t>(E)};
    const uint64_t st[1] = {static_cast<uint64_t>(d_h) * 2};
    const uint32_t bx[2] = {GT_BK, GT_BM}, bw[2] = {GT_BK, GT_BN};
    if (!encode_tma_map(&tm_x, cu_dt, 2, x, dx, st, bx, 1) || !encode_tma_map(&tm_w, cu_dt, 2, wg, dw, st, bw, 1))
        return cudaErrorInvalidValue;
    GateTcParams p;
    p.part = part;
    p.wnorm = wnorm;
    p.xss = xss;
    p.wg = static_cast<const uint8_t *>(wg);
    p.T = static_cast<int>(T);
    p.E = static_cast<int>(E);
    p.d_h = static_cast<int>(d_h);
    p.nk = nk;
    p.ks = ks;
    p.err = err;

    static std::atomic<bool> attr_done[64];  // zero-initialised; several host threads may launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const size_t sel_smem = select_smem_bytes(d_h, E);
    const int slots = static_cast<int>((E + 31) / 32);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gate_tc_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, GT_SMEM);
        if (e != cudaSuccess) return e;
#define MOE_SEL_ATTR(SL)                                                                                 \
        e = cudaFuncSetAttribute(gate_select_kernel<DT, SL>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 kGateTcMaxSelectSmem);                                                  \
        if (e != cudaSuccess) return e;
        MOE_SEL_ATTR(2)
        MOE_SEL_ATTR(4)
        MOE_SEL_ATTR(8)
        MOE_SEL_ATTR(16)
        MOE_SEL_ATTR(32)
#undef MOE_SEL_ATTR
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    const dim3 grid(static_cast<unsigned>((T + GT_BM - 1) / GT_BM), static_cast<unsigned>((E + GT_BN - 1) / GT_BN),
                    static_cast<unsigned>(S));
    // the partials leave by tensor stores when each token row of them is a
    // whole number of 16-byte units (E % 4 == 0); [E, T, S] so that the rows
    // of a tile past T are clipped in every split
    CUtensorMap tm_p = tm_x;
    p.tma_store = 0;
    if (E % 4 == 0) {
        const uint64_t dp[3] = {static_cast<uint64_t>(E), static_cast<uint64_t>(T), static_cast<uint64_t>(S)};
        const uint64_t sp[2] = {static_cast<uint64_t>(E) * 4, static_cast<uint64_t>(T) * E * 4};
        const uint32_t bp[3] = {32, GT_BM, 1};
        if (encode_tma_map(&tm_p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, part, dp, sp, bp, 1)) p.tma_store = 1;
        else tm_p = tm_x;
    }
    cudaError_t e = launch_pdl(gate_tc_kernel<DT>, grid, dim3(GT_THREADS), GT_SMEM, stream, tm_x, tm_w, tm_p, p);
    if (e != cudaSuccess) return e;

    // |logit~ - logit| <= coef * (|x| |w| + |bias|) + 2^-22 |logit~|
    const double u = std::ldexp(1.0, -24);
    const double groups = 4.0 * ks;                           // K=16 MMA steps per split
    const double c_tc = 18.0 * groups * 2.0 * u;              // tensor-core splits
    const double c_fixed = (static_cast<double>(d_h) / 32.0 + 6.0) * u;  // fixed-order sum
    const double c_sum = (S + 2.0) * u;                       // partials and bias
    const double norms = (1.0 + std::ldexp(1.0, -9)) * (1.0 + std::ldexp(1.0, -9));  // fp32 norms
    const float coef = static_cast<float>(2.0 * (c_tc + c_fixed + c_sum) * norms);
    const unsigned sel_grid = static_cast<unsigned>((T + SEL_WARPS - 1) / SEL_WARPS);
#define MOE_SEL_CASE(SL)                                                                                     \
    if (slots <= SL)                                                                                         \
        return launch_pdl(gate_select_kernel<DT, SL>, dim3(sel_grid), dim3(SEL_WARPS * 32), sel_smem, stream, \
                          static_cast<const uint8_t *>(x), static_cast<const uint8_t *>(wg), bias,           \
                          static_cast<const float *>(part), static_cast<const float *>(wnorm),               \
                          static_cast<const float *>(xss), static_cast<int>(T), static_cast<int>(E),         \
                          static_cast<int>(d_h), S,                                                          \
                          static_cast<int>(k), coef, logits, topk_idx, topk_w);
    MOE_SEL_CASE(2)
    MOE_SEL_CASE(4)
    MOE_SEL_CASE(8)
    MOE_SEL_CASE(16)
    MOE_SEL_CASE(32)
#undef MOE_SEL_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

bool gate_tc_applies(int64_t T, int64_t d_h, int64_t E) {
    return T >= kGateTcMinTokens && d_h % GT_BK == 0 && E <= 1024 &&
           select_smem_bytes(d_h, E) <= static_cast<size_t>(kGateTcMaxSelectSmem);
}

size_t gate_tc_scratch_bytes(int64_t T, int64_t E) {
    if (T < kGateTcMinTokens) return 0;
    const size_t part = static_cast<size_t>(splits_for(T, E)) * T * E * 4;
    return (part + 255) / 256 * 256 + (static_cast<size_t>(E) * 4 + 255) / 256 * 256 +
           (static_cast<size_t>(splits_for(T, E)) * T * 4 + 255) / 256 * 256;
}

cudaError_t launch_gate_tc(const void *x, const void *wg, const float *bias, int64_t T, int64_t d_h,
                           int64_t E, int64_t k, int dtype, float *logits, void *scratch,
                           int32_t *topk_idx, float *topk_w, int32_t *err, cudaStream_t stream) {
    float *part = static_cast<float *>(scratch);
    const size_t part_bytes = static_cast<size_t>(splits_for(T, E)) * T * E * 4;
    float *wnorm = reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) + (part_bytes + 255) / 256 * 256);
    float *xss = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(wnorm) +
                                           (static_cast<size_t>(E) * 4 + 255) / 256 * 256);
    if (dtype == kBF16)
        return launch_typed<kBF16>(x, wg, bias, T, d_h, E, k, logits, part, wnorm, xss, topk_idx, topk_w, err,
                                   stream);
    return launch_typed<kF16>(x, wg, bias, T, d_h, E, k, logits, part, wnorm, xss, topk_idx, topk_w, err,
                              stream);
}

}  // namespace moe

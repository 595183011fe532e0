// gate_topk.cu -- gate logits, top-k selection and softmax weights.
//
// The pages call the gate (CSDN "forward", step 1: expert_indices,
// expert_scores = gating_network(x)) but do not print it.  This library reads
// it as a linear gate with softmax over fp32 logits, top-k with ties to the
// lower expert id, and the top-k probabilities as the routing weights.
//
// Logit summation order (fixed, so the routing is reproducible bit for bit):
// the d_hidden axis is cut into 8-element chunks; chunk c is summed by warp
// lane (c mod 32) in ascending index with fmaf, then the 32 lane partials are
// combined by the xor butterfly s = 16, 8, 4, 2, 1.  The kernel is the
// natural warp-split-K dot product: a warp owns a (4 or 8)-token x 8-expert tile,
// each lane keeps one partial per (token, expert) pair and reads its 16-byte
// chunk of every row from shared memory (conflict free); 256-element slices
// of x and W_g arrive by TMA (one box of token rows and one of expert rows per
// slice) in a 4-stage ring.
//
// Three shapes of the same kernel:
//   * E <= 64: one CTA holds 1 token (small batches) or 4 tokens x all
//     experts and also selects the top-k from its logits in shared memory
//     (one launch for the gate);
//   * many tokens: CTA = 16 tokens x 16 experts (4 warps of 8 x 8 pairs), then
//     topk_softmax_kernel;
//   * few tokens: CTA = one warp of 4 tokens x 8 experts (more CTAs in
//     flight), then topk_softmax_kernel.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int SLICE = 256;                // elements per lane round: 32 lanes x 8
constexpr int ROW_BYTES = SLICE * 2;      // 512 B of one row per slice
// Ring depth: the small-batch shapes keep up to 8 slices (about 200 KB) in
// flight, since their time is the latency of the first slices; the 4-warp
// many-token shape keeps 4 (three CTAs per SM, each 64 KB of ring).  Measured
// at 4096 tokens x 256 experts x 7168: 3, 4 or 6 stages and one to three CTAs
// per SM within 10%, 16 x 16 fastest among 8x16 / 16x16 / 16x32 / 32x16 tiles;
// 8 x 8 pairs per warp 2% faster than 4 x 8 (300 vs 306 us; 8x16 and 16x8
// CTAs of 8 x 8 warps 340-357 us, 32x16 and 16x32 ones 304 us).
__host__ __device__ constexpr int gate_stages(int rows, bool many_tokens) {
    return many_tokens ? 4 : ((200 * 1024) / (rows * ROW_BYTES) > 8 ? 8 : (200 * 1024) / (rows * ROW_BYTES));
}

// Top-k by (logit desc, id asc) and the softmax weights of TOK tokens whose
// 64 logits per token (E <= 64 valid) sit in shared memory, lsm[TOK][64],
// with every thread of the CTA taking part (the single-token latency case).
// Q = NT / (TOK * 64) threads rank one value, each against 64 / Q of the
// token's values (4-wide shared loads, a short loop), and their counts are
// added by shuffles; the value of rank r < k is selection slot r.  The
// softmax denominator is summed by the token's warp as in warp_topk_rounds
// (per lane: its expert, then expert + 32; then the xor butterfly), so the
// weights are the same bits either way.  Scratch after lsm: ranks and the
// top logit per token.
template <int TOK, int NT>
__device__ __forceinline__ void cta_topk_softmax(float *lsm, int t0, int T, int E, int k,
                                                 int32_t *__restrict__ topk_idx,
                                                 float *__restrict__ topk_w) {
    constexpr int EXP = 64, Q = NT / (TOK * EXP), PER = EXP / Q;
    static_assert(Q >= 1 && Q * TOK * EXP == NT && PER % 4 == 0, "ranking shape");
    int *rank_s = reinterpret_cast<int *>(lsm + TOK * EXP);
    float *top_s = reinterpret_cast<float *>(rank_s + TOK * EXP);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vi = tid / Q, part = tid - vi * Q;
    const int tt = vi / EXP, e = vi - tt * EXP;
    const float mine = lsm[vi];
    const float4 *row4 = reinterpret_cast<const float4 *>(lsm + tt * EXP + part * PER);
    int r = 0;
#pragma unroll 1
    for (int q = 0; q < PER / 4; ++q) {
        const float4 o = row4[q];
        const int o0 = part * PER + q * 4;
        r += (o0 < E && (o.x > mine || (o.x == mine && o0 < e))) ? 1 : 0;
        r += (o0 + 1 < E && (o.y > mine || (o.y == mine && o0 + 1 < e))) ? 1 : 0;
        r += (o0 + 2 < E && (o.z > mine || (o.z == mine && o0 + 2 < e))) ? 1 : 0;
        r += (o0 + 3 < E && (o.w > mine || (o.w == mine && o0 + 3 < e))) ? 1 : 0;
    }
#pragma unroll
    for (int sh = 1; sh < Q; sh <<= 1) r += __shfl_xor_sync(0xffffffffu, r, sh);
    if (part == 0) {
        rank_s[vi] = r;
        if (e < E && r == 0) top_s[tt] = mine;
    }
    __syncthreads();
    const int t = t0 + warp;
    if (warp < TOK && t < T) {
        const float top = top_s[warp];
        const float v0 = lsm[warp * EXP + lane], v1 = lsm[warp * EXP + 32 + lane];
        float sum = 0.0f;
        if (lane < E) sum += expf(v0 - top);
        if (32 + lane < E) sum += expf(v1 - top);
#pragma unroll
        for (int sh = 16; sh >= 1; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
        const int r0 = rank_s[warp * EXP + lane], r1 = rank_s[warp * EXP + 32 + lane];
        int32_t *idx_out = topk_idx + static_cast<int64_t>(t) * k;
        float *w_out = topk_w + static_cast<int64_t>(t) * k;
        if (lane < E && r0 < k) {
            idx_out[r0] = lane;
            w_out[r0] = expf(v0 - top) / sum;
        }
        if (32 + lane < E && r1 < k) {
            idx_out[r1] = 32 + lane;
            w_out[r1] = expf(v1 - top) / sum;
        }
    }
}

// Warp argmax by (logit desc, id asc) over k rounds, then the softmax weights
// (for many experts: k rounds cost less than ranking every value).
// Lane holds v[s] = logit of expert s*32 + lane (or -inf past E).
template <int SLOTS>
__device__ __forceinline__ void warp_topk_rounds(float (&v)[SLOTS], int E, int k, int32_t *idx_out,
                                                 float *w_out, int lane) {
    bool taken[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) taken[s] = s * 32 + lane >= E;
    float top_logit = 0.0f, my_logit = 0.0f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
        float best = -INFINITY;
        int best_id = 0x7fffffff;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const int e = s * 32 + lane;
            if (!taken[s] && (best_id == 0x7fffffff || v[s] > best || (v[s] == best && e < best_id))) {
                best = v[s];
                best_id = e;
            }
        }
#pragma unroll
        for (int sh = 16; sh >= 1; sh >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, sh);
            const int oid = __shfl_xor_sync(0xffffffffu, best_id, sh);
            if (oid != 0x7fffffff && (best_id == 0x7fffffff || ob > best || (ob == best && oid < best_id))) {
                best = ob;
                best_id = oid;
            }
        }
#pragma unroll
        for (int s = 0; s < SLOTS; ++s)
            if (s * 32 + lane == best_id) taken[s] = true;
        if (j == 0) top_logit = best;
        if (j == lane) {
            my_logit = best;
            my_id = best_id;
        }
    }
    float sum = 0.0f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s)
        if (s * 32 + lane < E) sum += expf(v[s] - top_logit);
#pragma unroll
    for (int sh = 16; sh >= 1; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
    if (lane < k) {
        idx_out[lane] = my_id;
        w_out[lane] = expf(my_logit - top_logit) / sum;
    }
}

template <int DT, int TPW, int WT, int WE, bool FUSE_TOPK>
__global__ void __launch_bounds__(WT *WE * 32)
    gate_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const float *__restrict__ bias, int T, int d_h, int E, int k,
                float *__restrict__ logits, int32_t *__restrict__ topk_idx,
                float *__restrict__ topk_w) {
    constexpr int TOK = WT * TPW, EXP = WE * 8, ROWS = TOK + EXP;
    constexpr int STAGE_BYTES = ROWS * ROW_BYTES;
    constexpr int GATE_STAGES = gate_stages(ROWS, WT * WE > 1 && !FUSE_TOPK);
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * TOK, e0 = blockIdx.y * EXP;
    const int wt = (warp / WE) * TPW;  // warp's first token in the tile
    const int we = (warp % WE) * 8;  // warp's first expert in the tile
    const int n_slices = d_h / SLICE;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + GATE_STAGES * STAGE_BYTES);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + GATE_STAGES);

    // one slice = a 256-column box of the CTA's token rows and expert rows,
    // two TMA copies landing on the stage's mbarrier (rows past T / E read 0)
    auto load_slice = [&](int s) {
        const int st = s % GATE_STAGES;
        uint8_t *stage = smem + st * STAGE_BYTES;
        const uint32_t bar = smem_u32(full + st);
        mbar_arrive_expect_tx(bar, STAGE_BYTES);
        tma_load_2d(smem_u32(stage), &tm_x, bar, s * SLICE, t0);
        tma_load_2d(smem_u32(stage + TOK * ROW_BYTES), &tm_w, bar, s * SLICE, e0);
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < GATE_STAGES; ++i) mbar_init(smem_u32(full + i), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    __syncthreads();

    float acc[TPW][8];
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    griddep_wait();  // x (and W_g) may come from the previous kernel
    griddep_launch_dependents();

    if (threadIdx.x == 0)
        for (int s = 0; s < GATE_STAGES && s < n_slices; ++s) load_slice(s);
    int done = 0;  // slices consumed
    for (int s = 0; s < n_slices; ++s) {
        // every thread waits for the stage (bounded; a lost copy ends the loop)
        if (!mbar_wait_bounded(smem_u32(full + s % GATE_STAGES),
                               static_cast<uint32_t>((s / GATE_STAGES) & 1), abort_flag, nullptr))
            break;
        const uint8_t *stage = smem + (s % GATE_STAGES) * STAGE_BYTES;
        // lane owns chunk `lane` of the slice: elements 8*lane .. 8*lane+7, ascending
        uint4 xv[TPW], wv[8];
#pragma unroll
        for (int i = 0; i < TPW; ++i)
            xv[i] = *reinterpret_cast<const uint4 *>(stage + (wt + i) * ROW_BYTES + lane * 16);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            wv[j] = *reinterpret_cast<const uint4 *>(stage + (TOK + we + j) * ROW_BYTES + lane * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t xw[TPW], ww[8];
#pragma unroll
            for (int i = 0; i < TPW; ++i)
                xw[i] = q == 0 ? xv[i].x : q == 1 ? xv[i].y : q == 2 ? xv[i].z : xv[i].w;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ww[j] = q == 0 ? wv[j].x : q == 1 ? wv[j].y : q == 2 ? wv[j].z : wv[j].w;
            // element 2q of every pair, then element 2q+1: the two updates of
            // one accumulator are TPW*8 independent FMAs apart
#pragma unroll
            for (int i = 0; i < TPW; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fma_mixed<DT, false>(xw[i], ww[j], acc[i][j]);
#pragma unroll
            for (int i = 0; i < TPW; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fma_mixed<DT, true>(xw[i], ww[j], acc[i][j]);
        }
        __syncthreads();  // every warp is done with this stage: refill it
        if (threadIdx.x == 0 && s + GATE_STAGES < n_slices && !*abort_flag) load_slice(s + GATE_STAGES);
        done = s + 1;
    }
    if (threadIdx.x == 0) {
        // after a timeout, let the copies still in flight land before exit
        for (int s = done; s < n_slices && s < done + GATE_STAGES; ++s) {
            const unsigned long long t_start = global_timer_ns();
            while (!mbar_try_wait(smem_u32(full + s % GATE_STAGES), static_cast<uint32_t>((s / GATE_STAGES) & 1)))
                if (global_timer_ns() - t_start > kWaitTimeoutNs) break;
        }
    }

    // xor butterfly s = 16, 8, 4, 2, 1; every lane ends with the full sum
#pragma unroll
    for (int i = 0; i < TPW; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float v = acc[i][j];
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, sh);
            acc[i][j] = v;
        }

    // every lane now holds all TPW*8 sums; lane L keeps pairs L, L + 32, ...
    // and writes them: one select chain and one store per pair
    if constexpr (!FUSE_TOPK) {
#pragma unroll
        for (int r = 0; r < (TPW * 8 + 31) / 32; ++r) {
            const int pr = r * 32 + lane;
            float mine = 0.0f;
#pragma unroll
            for (int i = 0; i < TPW; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) mine = (i * 8 + j == pr) ? acc[i][j] : mine;
            const int my_t = t0 + wt + (pr >> 3), my_e = e0 + we + (pr & 7);
            if (pr < TPW * 8 && my_t < T && my_e < E) {
                float l = mine;
                if (bias) l = l + bias[my_e];
                logits[static_cast<int64_t>(my_t) * E + my_e] = l;
            }
        }
    } else {
        static_assert(TPW * 8 <= 32, "one pair per lane");
        float mine = 0.0f;
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) mine = (i * 8 + j == lane) ? acc[i][j] : mine;
        const int my_i = lane >> 3, my_j = lane & 7;
        const int my_t = t0 + wt + my_i, my_e = e0 + we + my_j;
        // one CTA holds every expert of its TOK tokens: logits to shared
        // memory, then warp w selects the top-k of token t0 + w
        static_assert(!FUSE_TOPK || (WT == 1 && EXP == 64 && TPW <= WE), "fused shape");
        __syncthreads();  // the ring is no longer read
        float *lsm = reinterpret_cast<float *>(smem);  // [TOK][EXP]
        if (lane < TPW * 8) {
            float l = mine;
            if (my_e < E && bias) l = l + bias[my_e];
            lsm[(wt + my_i) * EXP + we + my_j] = l;
            if (my_t < T && my_e < E) logits[static_cast<int64_t>(my_t) * E + my_e] = l;
        }
        __syncthreads();
        cta_topk_softmax<TOK, WT * WE * 32>(lsm, t0, T, E, k, topk_idx, topk_w);
    }
}

// One warp per token over logits in global memory.
constexpr int TK_WARPS = 8;

template <int SLOTS>
__global__ void __launch_bounds__(TK_WARPS * 32)
    topk_softmax_kernel(const float *__restrict__ logits, int T, int E, int k,
                        int32_t *__restrict__ topk_idx, float *__restrict__ topk_w) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * TK_WARPS + warp;
    griddep_wait();
    griddep_launch_dependents();
    if (t >= T) return;
    const float *row = logits + static_cast<int64_t>(t) * E;
    float v[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int e = s * 32 + lane;
        v[s] = e < E ? row[e] : -INFINITY;
    }
    warp_topk_rounds<SLOTS>(v, E, k, topk_idx + static_cast<int64_t>(t) * k,
                             topk_w + static_cast<int64_t>(t) * k, lane);
}

template <int DT, int TPW, int WT, int WE, bool FUSE>
cudaError_t launch_gate_shape(const void *x, const void *wg, const float *bias, int64_t T,
                              int64_t d_h, int64_t E, int64_t k, float *logits, int32_t *idx,
                              float *w, cudaStream_t stream) {
    constexpr int TOK = WT * TPW, EXP = WE * 8;
    constexpr int GATE_STAGES = gate_stages(TOK + EXP, WT * WE > 1 && !FUSE);
    const size_t smem = static_cast<size_t>(GATE_STAGES) * (TOK + EXP) * ROW_BYTES + 8 * GATE_STAGES + 16;
    CUtensorMap tm_x, tm_w;
    if (!encode_tma_2d_plain(&tm_x, x, static_cast<uint64_t>(d_h), static_cast<uint64_t>(T), SLICE, TOK) ||
        !encode_tma_2d_plain(&tm_w, wg, static_cast<uint64_t>(d_h), static_cast<uint64_t>(E), SLICE, EXP))
        return cudaErrorInvalidValue;
    auto kern = gate_kernel<DT, TPW, WT, WE, FUSE>;
    static std::atomic<bool> attr_done[64];  // zero-initialised; several host threads may launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (smem > 48 * 1024 && (dev < 0 || dev >= 64 || !attr_done[dev])) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    dim3 grid(static_cast<unsigned>((T + TOK - 1) / TOK), static_cast<unsigned>((E + EXP - 1) / EXP));
    return launch_pdl(kern, grid, dim3(WT * WE * 32), smem, stream, tm_x, tm_w, bias, (int)T,
                      (int)d_h, (int)E, (int)k, logits, idx, w);
}

cudaError_t launch_topk(const float *logits, int64_t T, int64_t E, int64_t k, int32_t *topk_idx,
                        float *topk_w, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>((T + TK_WARPS - 1) / TK_WARPS);
    const int slots = static_cast<int>((E + 31) / 32);
#define MOE_TOPK_CASE(S)                                                                        \
    if (slots <= S)                                                                             \
        return launch_pdl(topk_softmax_kernel<S>, dim3(grid), dim3(TK_WARPS * 32), 0, stream,    \
                          logits, (int)T, (int)E, (int)k, topk_idx, topk_w);
    MOE_TOPK_CASE(2)
    MOE_TOPK_CASE(4)
    MOE_TOPK_CASE(8)
    MOE_TOPK_CASE(16)
    MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
    return cudaErrorInvalidValue;
}

template <int DT>
cudaError_t launch_gate_typed(const void *x, const void *wg, const float *bias, int64_t T,
                              int64_t d_h, int64_t E, int64_t k, float *logits, int32_t *idx,
                              float *w, cudaStream_t stream) {
    // E <= 64: one CTA holds all experts of its tokens (8 warps x 8 experts)
    // and selects their top-k; one token per CTA while that still fills the
    // GPU with few CTAs, else 4 tokens per CTA
    if (E <= 64) {
        if (T <= 4 * device_sm_count())
            return launch_gate_shape<DT, 1, 1, 8, true>(x, wg, bias, T, d_h, E, k, logits, idx, w, stream);
        return launch_gate_shape<DT, 4, 1, 8, true>(x, wg, bias, T, d_h, E, k, logits, idx, w, stream);
    }
    cudaError_t e;
    if (T >= 512)  // 16 tokens x 16 experts per CTA: 4 warps of 8 x 8 pairs, three CTAs per SM
        e = launch_gate_shape<DT, 8, 2, 2, false>(x, wg, bias, T, d_h, E, k, logits, idx, w, stream);
    else           // one warp of 4 x 8 pairs per CTA
        e = launch_gate_shape<DT, 4, 1, 1, false>(x, wg, bias, T, d_h, E, k, logits, idx, w, stream);
    if (e != cudaSuccess) return e;
    return launch_topk(logits, T, E, k, idx, w, stream);
}

}  // namespace

cudaError_t launch_gate_topk(const void *x, const void *wg, const float *bias, int64_t T,
                             int64_t d_h, int64_t E, int64_t k, int dtype, float *logits,
                             int32_t *topk_idx, float *topk_w, void *tc_scratch, int32_t *err,
                             cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    // many tokens: logits on the tensor cores, the routing made exact by the
    // fixed-order recompute of every candidate (gate_tc.cu)
    if (tc_scratch != nullptr && gate_tc_applies(T, d_h, E))
        return launch_gate_tc(x, wg, bias, T, d_h, E, k, dtype, logits, tc_scratch, topk_idx, topk_w, err,
                              stream);
    if (dtype == kBF16)
        return launch_gate_typed<kBF16>(x, wg, bias, T, d_h, E, k, logits, topk_idx, topk_w, stream);
    return launch_gate_typed<kF16>(x, wg, bias, T, d_h, E, k, logits, topk_idx, topk_w, stream);
}

}  // namespace moe

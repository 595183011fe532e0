// gate_topk.cu -- gate logits, top-k selection and softmax weights.
//
// The pages call the gate (CSDN "forward", step 1: expert_indices,
// expert_scores = gating_network(x)) but do not print it.  This build reads
// it as a linear gate with softmax over fp32 logits, top-k with ties to the
// lower expert id, and the top-k probabilities as the routing weights.
//
// Logit summation order (fixed, so the routing is reproducible bit for bit):
// the d_hidden axis is cut into 8-element chunks; chunk c is summed by warp
// lane (c mod 32) in ascending index with fmaf, then the 32 lane partials are
// combined by the xor butterfly s = 16, 8, 4, 2, 1.  The kernel is the
// natural warp-split-K dot product: a warp owns an 8-token x 8-expert tile,
// each lane keeps one partial per (token, expert) pair, and 256-element
// slices of x and W_g are staged through shared memory with cp.async.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int GT_TOK = 16;        // tokens per CTA
constexpr int GT_EXP = 32;        // experts per CTA
constexpr int WT_TOK = 8;         // tokens per warp
constexpr int WT_EXP = 8;         // experts per warp
constexpr int GT_WARPS = (GT_TOK / WT_TOK) * (GT_EXP / WT_EXP);  // 8
constexpr int GT_THREADS = GT_WARPS * 32;
constexpr int SLICE = 256;        // elements per lane round: 32 lanes x 8
constexpr int ROW_BYTES = SLICE * 2;  // 512 B of one row per slice

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
    const int n = pred ? 16 : 0;  // zero-fill rows past the end
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int DT>
__global__ void __launch_bounds__(GT_THREADS)
    gate_logits_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ wg,
                       const float *__restrict__ bias, int T, int d_h, int E,
                       float *__restrict__ logits) {
    // [2 buffers][GT_TOK + GT_EXP rows][512 B]
    __shared__ __align__(16) uint8_t tiles[2][GT_TOK + GT_EXP][ROW_BYTES];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * GT_TOK, e0 = blockIdx.y * GT_EXP;
    const int wt = (warp / (GT_EXP / WT_EXP)) * WT_TOK;  // warp's token offset in the tile
    const int we = (warp % (GT_EXP / WT_EXP)) * WT_EXP;  // warp's expert offset
    const int n_slices = d_h / SLICE;

    // one slice = (GT_TOK + GT_EXP) rows x 32 chunks of 16 B = 1536 chunks
    auto load_slice = [&](int s, int buf) {
        for (int c = threadIdx.x; c < (GT_TOK + GT_EXP) * 32; c += GT_THREADS) {
            const int r = c >> 5, ch = c & 31;
            const bool is_tok = r < GT_TOK;
            const int gr = is_tok ? t0 + r : e0 + (r - GT_TOK);
            const bool ok = is_tok ? gr < T : gr < E;
            const uint16_t *base = is_tok ? x : wg;
            const uint16_t *src = base + static_cast<int64_t>(ok ? gr : 0) * d_h + s * SLICE + ch * 8;
            cp_async16(smem_u32(&tiles[buf][r][ch * 16]), src, ok);
        }
        cp_async_commit();
    };

    float acc[WT_TOK][WT_EXP];
#pragma unroll
    for (int i = 0; i < WT_TOK; ++i)
#pragma unroll
        for (int j = 0; j < WT_EXP; ++j) acc[i][j] = 0.0f;

    load_slice(0, 0);
    for (int s = 0; s < n_slices; ++s) {
        const int buf = s & 1;
        if (s + 1 < n_slices) {
            load_slice(s + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        // lane owns chunk `lane` of this slice: elements [8*lane, 8*lane + 8)
#pragma unroll
        for (int w = 0; w < 4; ++w) {  // 4 words = 8 elements, ascending
            float2 xv[WT_TOK], wv[WT_EXP];
#pragma unroll
            for (int i = 0; i < WT_TOK; ++i)
                xv[i] = unpack2<DT>(*reinterpret_cast<const uint32_t *>(&tiles[buf][wt + i][lane * 16 + w * 4]));
#pragma unroll
            for (int j = 0; j < WT_EXP; ++j)
                wv[j] = unpack2<DT>(*reinterpret_cast<const uint32_t *>(&tiles[buf][GT_TOK + we + j][lane * 16 + w * 4]));
#pragma unroll
            for (int i = 0; i < WT_TOK; ++i)
#pragma unroll
                for (int j = 0; j < WT_EXP; ++j) {
                    acc[i][j] = fmaf(xv[i].x, wv[j].x, acc[i][j]);
                    acc[i][j] = fmaf(xv[i].y, wv[j].y, acc[i][j]);
                }
        }
        __syncthreads();
    }

    // xor butterfly s = 16, 8, 4, 2, 1; every lane ends with the full sum
#pragma unroll
    for (int i = 0; i < WT_TOK; ++i)
#pragma unroll
        for (int j = 0; j < WT_EXP; ++j) {
            float v = acc[i][j];
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, sh);
            acc[i][j] = v;
        }
    // lane L writes pairs L and L + 32 of the warp's 64
#pragma unroll
    for (int i = 0; i < WT_TOK; ++i)
#pragma unroll
        for (int j = 0; j < WT_EXP; ++j) {
            const int pair = i * WT_EXP + j;
            if ((pair & 31) == lane) {
                const int t = t0 + wt + i, e = e0 + we + j;
                if (t < T && e < E) {
                    float l = acc[i][j];
                    if (bias) l = l + bias[e];
                    logits[static_cast<int64_t>(t) * E + e] = l;
                }
            }
        }
}

// One warp per token.  Each lane holds E/32 logits (expert e at lane e % 32,
// slot e / 32).  k rounds of a warp argmax by (logit desc, id asc); softmax
// over all E in fp32 with the max subtracted.
constexpr int TK_WARPS = 8;

template <int SLOTS>
__global__ void __launch_bounds__(TK_WARPS * 32)
    topk_softmax_kernel(const float *__restrict__ logits, int T, int E, int k,
                        int32_t *__restrict__ topk_idx, float *__restrict__ topk_w) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * TK_WARPS + warp;
    if (t >= T) return;
    const float *row = logits + static_cast<int64_t>(t) * E;
    float v[SLOTS];
    bool taken[SLOTS];
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int e = s * 32 + lane;
        v[s] = e < E ? row[e] : -INFINITY;
        taken[s] = e >= E;
    }
    float top_logit = 0.0f;
    float sel_logit[32];
    int sel_id[32];
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
        sel_logit[j] = best;
        sel_id[j] = best_id;
        if (j == 0) top_logit = best;
    }
    float sum = 0.0f;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s)
        if (s * 32 + lane < E) sum += expf(v[s] - top_logit);
#pragma unroll
    for (int sh = 16; sh >= 1; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
    if (lane < k) {
        float l = 0.0f;
        int id = 0;
        for (int j = 0; j < k; ++j)
            if (j == lane) {
                l = sel_logit[j];
                id = sel_id[j];
            }
        topk_idx[static_cast<int64_t>(t) * k + lane] = id;
        topk_w[static_cast<int64_t>(t) * k + lane] = expf(l - top_logit) / sum;
    }
}

}  // namespace

cudaError_t launch_gate_logits(const void *x, const void *wg, const float *bias, int64_t T,
                               int64_t d_h, int64_t E, int dtype, float *logits,
                               cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>((T + GT_TOK - 1) / GT_TOK),
              static_cast<unsigned>((E + GT_EXP - 1) / GT_EXP));
    const auto *xp = static_cast<const uint16_t *>(x);
    const auto *wp = static_cast<const uint16_t *>(wg);
    if (dtype == kBF16)
        gate_logits_kernel<kBF16><<<grid, GT_THREADS, 0, stream>>>(xp, wp, bias, (int)T, (int)d_h, (int)E, logits);
    else
        gate_logits_kernel<kF16><<<grid, GT_THREADS, 0, stream>>>(xp, wp, bias, (int)T, (int)d_h, (int)E, logits);
    return cudaGetLastError();
}

cudaError_t launch_topk_softmax(const float *logits, int64_t T, int64_t E, int64_t k,
                                int32_t *topk_idx, float *topk_w, cudaStream_t stream) {
    if (T <= 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((T + TK_WARPS - 1) / TK_WARPS);
    const int slots = static_cast<int>((E + 31) / 32);
#define MOE_TOPK_CASE(S)                                                                        \
    if (slots <= S) {                                                                           \
        topk_softmax_kernel<S><<<grid, TK_WARPS * 32, 0, stream>>>(logits, (int)T, (int)E, (int)k, \
                                                                    topk_idx, topk_w);          \
        return cudaGetLastError();                                                              \
    }
    MOE_TOPK_CASE(1)
    MOE_TOPK_CASE(2)
    MOE_TOPK_CASE(4)
    MOE_TOPK_CASE(8)
    MOE_TOPK_CASE(16)
    MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
    return cudaErrorInvalidValue;
}

}  // namespace moe

// internal.h -- host-side launchers of the kernels (C++ linkage, not exported).
// The C-ABI layer validates every argument before calling these.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda.h>

namespace moe {

int device_sm_count();
// capi.cu: CTAs of a persistent expert-MLP launch with `tiles` tiles: one per
// SM (at most `tiles`), or the MOE_MLP_GRID environment variable's count
int mlp_grid(int64_t tiles);

// grouped_gemm.cu: tensor map of a row-major [rows, inner] 16-bit matrix,
// box = box_inner x box_rows elements, no swizzle.  False if encoding fails.
bool encode_tma_2d_plain(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows,
                         uint32_t box_inner, uint32_t box_rows);
// grouped_gemm.cu: any tensor map (CUtensorMapDataType in data_type); dims,
// box innermost first; strides in bytes for dims 1..rank-1; 128-byte swizzle
// or none.  False if encoding fails.
bool encode_tma_map(CUtensorMap *m, int data_type, int rank, const void *ptr, const uint64_t *dims,
                    const uint64_t *strides_bytes, const uint32_t *box, int swizzle_128b);

// gate_topk.cu: logits (written to `logits`, [T, E] fp32), top-k ids and
// weights.  tc_scratch (gate_tc_scratch_bytes(T, E) bytes, or null) lets
// many-token calls run the tensor-core path of gate_tc.cu; err (nullable)
// receives a timed-out wait of that path.
cudaError_t launch_gate_topk(const void *x, const void *wg, const float *bias, int64_t T,
                             int64_t d_h, int64_t E, int64_t k, int dtype, float *logits,
                             int32_t *topk_idx, float *topk_w, void *tc_scratch, int32_t *err,
                             cudaStream_t stream);

// gate_tc.cu: the tensor-core gate (tokens at least kGateTcMinTokens): its
// scratch (split-K partial logits and the gate rows' norms), whether it
// applies to a shape, and the launch (logits as launch_gate_topk writes them:
// the fixed-order value for every expert that could be selected, the
// tensor-core value for the others).
constexpr int64_t kGateTcMinTokens = 1024;
constexpr int kGateTcMaxSelectSmem = 200 * 1024;
size_t gate_tc_scratch_bytes(int64_t T, int64_t E);
bool gate_tc_applies(int64_t T, int64_t d_h, int64_t E);
cudaError_t launch_gate_tc(const void *x, const void *wg, const float *bias, int64_t T, int64_t d_h,
                           int64_t E, int64_t k, int dtype, float *logits, void *scratch,
                           int32_t *topk_idx, float *topk_w, int32_t *err, cudaStream_t stream);

// capi.cu: the host-side argument checks shared by both dispatch entry
// points (a moe_status_t value; MOE_OK when the call may go ahead).
int check_dispatch_args(const int32_t *topk_idx, int64_t T, int64_t k, int64_t E, int64_t block_m,
                        const int32_t *group_sizes, const int32_t *group_offsets,
                        const int32_t *group_padded_offsets, const int32_t *group_idx_for_bx,
                        const int32_t *sorted_token_idx, const float *sorted_row_weight,
                        const int32_t *token_topk_to_pos);

// dispatch.cu
size_t dispatch_scratch_bytes(int64_t n_pairs, int64_t E);
cudaError_t launch_dispatch(const int32_t *topk_idx, const float *topk_w, int64_t T, int64_t k,
                            int64_t E, int64_t block_m, int32_t *sizes, int32_t *offsets, int32_t *padded,
                            int32_t *gidx, int64_t m_blocks, int32_t *sorted_token_idx,
                            float *sorted_row_weight, int32_t *pos, void *scratch,
                            int32_t *ready, cudaStream_t stream);

// rows.cu
cudaError_t launch_copy(const void *src, void *dst, int64_t bytes, cudaStream_t stream);
// one thread polls *flag (system scope) until >= expected or timeout_ns pass
// (then *err = kErrTimeout)
cudaError_t launch_wait_flag(const int32_t *flag, int32_t expected, int64_t timeout_ns, int32_t *err,
                             cudaStream_t stream);
cudaError_t launch_gather_rows(const void *x, const int32_t *sorted_token_idx, int64_t n_rows,
                               int64_t d_h, int elem_bytes, void *a_out, cudaStream_t stream);
// the same rows written in token order: a_out[token_topk_to_pos[t, j]] = x[t]
// (k <= 32; positions outside [0, n_rows) skipped); x is read once; bulk
// copies through shared memory when a row fits (err, nullable, receives a
// timed-out wait)
cudaError_t launch_scatter_rows(const void *x, const int32_t *token_topk_to_pos, int64_t T, int64_t k,
                                int64_t n_rows, int64_t d_h, int elem_bytes, void *a_out, int32_t *err,
                                cudaStream_t stream);
// pos_early: the positions and weights were complete before the previous
// kernel started (moe_forward: the dispatch precedes the expert MLP), so the
// combine may read them before its dependency wait
cudaError_t launch_reduce_fused(const void *x, int64_t n_rows, const int32_t *pos,
                                const float *w, const float *x_sf, const float *sf, int64_t T,
                                int64_t K, int64_t H, int in_dtype, int out_dtype, void *out,
                                int32_t *err, cudaStream_t stream, bool pos_early = false);

// grouped_gemm.cu
cudaError_t launch_grouped_gemm(bool gate_up, int dtype, const void *a, const void *w0,
                                const void *w1, const int32_t *sizes, const int32_t *offsets,
                                const int32_t *padded, const int32_t *gidx, int64_t m_blocks,
                                const float *row_weights, int64_t n_rows, int64_t K, int64_t N,
                                int64_t E, void *out, int32_t *err, cudaStream_t stream);
// Stage 1 and stage 2 in one persistent launch; `ready` (m_blocks + 1 int32:
// the per-block counters, then the tile counter) must be zero when the
// kernel starts.  With gather_idx (every block at most 64 rows, as when
// T <= 64), stage 1 gathers its rows from x [T, d_h] by those indices and `a`
// is not read.
cudaError_t launch_grouped_mlp(int dtype, const void *a, const void *w_gate, const void *w_up,
                               const void *w_down, const int32_t *sizes, const int32_t *offsets,
                               const int32_t *padded, const int32_t *gidx, int64_t m_blocks,
                               const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                               int64_t E, void *h, void *y, int32_t *ready, int32_t *err,
                               cudaStream_t stream, const void *x = nullptr,
                               const int32_t *gather_idx = nullptr, int64_t T = 0);

// grouped_mlp2.cu: both stages on CTA pairs (tcgen05 cta_group::2) from
// pre-gathered rows, no row weight; `ready` as launch_grouped_mlp.  Applies
// when d_e % 256 == 0, d_h % 512 == 0 and the work units fit the in-kernel
// schedule (n_rows / 256 + E <= 512).
bool grouped_mlp2_applies(int64_t n_rows, int64_t d_h, int64_t d_e, int64_t E);
cudaError_t launch_grouped_mlp2(int dtype, const void *a, const void *w_gate, const void *w_up,
                                const void *w_down, const int32_t *sizes, const int32_t *offsets,
                                const int32_t *padded, int64_t m_blocks, int64_t n_rows, int64_t d_h,
                                int64_t d_e, int64_t E, void *h, void *y, int32_t *ready, int32_t *err,
                                cudaStream_t stream);
// capi.cu: false when MOE_MLP_PAIRS=0 (tests compare the one-SM form)
bool mlp_pairs_enabled();

// grouped_gemm_w4.cu: int4 weights [E, N, K], two per byte as the pages pack
// them, into the tiled layout the int4 kernels read (tiles of R output
// channels; R = 128 for W_gate / W_up, 256 for W_down); bytes of that layout
// (-1 for bad sizes; K % 64 == 0).
int64_t pack_int4_bytes(int64_t E, int64_t N, int64_t K, int R);
cudaError_t launch_pack_int4(const uint8_t *plain, int64_t E, int64_t N, int64_t K, int R, uint8_t *packed,
                             cudaStream_t stream);
// Both expert stages with int4 weights (tiled by launch_pack_int4) and
// optional fp32 scales per output channel; stage-1 rows gathered from x
// [T, d_h] by gather_idx; the kernel works on units of at most 64 rows (a
// block with more rows is two units); `ready` (m_blocks + 1 int32) zero at
// kernel start.
cudaError_t launch_grouped_mlp_w4(int dtype, const void *x, const int32_t *gather_idx, int64_t T,
                                  const uint8_t *q_gate, const uint8_t *q_up, const uint8_t *q_down,
                                  const float *s_gate, const float *s_up, const float *s_down,
                                  const int32_t *sizes, const int32_t *offsets,
                                  const int32_t *padded, const int32_t *gidx, int64_t m_blocks,
                                  const float *row_weights, int64_t n_rows, int64_t d_h,
                                  int64_t d_e, int64_t E, void *h, void *y, int32_t *ready,
                                  int32_t *err, cudaStream_t stream);

// W4A8 (int4 weights x int8 activations, int32 sums) on the int4 kernel's
// stage-2 path: the int8 rows are widened to fp16 (exact) into rows_f16
// [n_rows, K], then every 256-channel tile sums one K chunk of at most
// kW4a8MaxChunkSub 64-wide sub-steps in fp32 (exact: every partial sum is an
// integer of magnitude <= 1024 * 16384 = 2^24) and stores (one chunk) or adds
// (several, integer atomics) its int32 results at m * ld_row + n * ld_col.
// dense_rows > 0: one block of that many rows (<= 64) and weight 0, no
// tables; otherwise the dispatch tables (64-row units as the expert MLP).
// counters: (blocks + 1) int32 and, when K is split, out (out_elems int32)
// are zeroed by the row kernel, ahead of the GEMM.  K % 64 == 0.
constexpr int64_t kW4a8MaxChunkSub = 256;
struct W4a8Plan {
    int64_t ksplit = 1, kchunk = 1;  // K chunks per tile and their sub-steps
};
W4a8Plan w4a8_plan(int64_t blocks, int64_t N, int64_t K);
cudaError_t launch_gemm_w4a8(const int8_t *x, const int32_t *gather_idx, int64_t T, const uint8_t *B,
                             const int32_t *sizes, const int32_t *offsets, const int32_t *padded,
                             const int32_t *gidx, int64_t m_blocks, int64_t dense_rows, int64_t n_rows,
                             int64_t N, int64_t K, void *rows_f16, int32_t *counters, int32_t *out,
                             int64_t ld_row, int64_t ld_col, int64_t out_elems, int32_t *err,
                             cudaStream_t stream);

}  // namespace moe

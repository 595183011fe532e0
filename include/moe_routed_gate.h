/*
 * moe_routed_gate.h -- C-ABI of the GB300 (sm_103a) routed-expert MoE forward.
 *
 * The forward of one DeepSeek-style MoE layer's routed experts:
 *   gate logits -> softmax / top-k -> counting-sort dispatch (four tables plus
 *   the sorted token-index and row-weight arrays, every expert padded to
 *   block_m = 128 rows) -> grouped gate/up GEMM with SiLU(gate)*up fused ->
 *   grouped down GEMM -> moe_reduce_fused combine.
 * Sources: the CSDN article "tilelang baseline" of the tilelang-metax MoE
 * contest operator (sections "forward", "stage 1 gate+up", "stage 2 down"),
 * the TileLang tutorial ch.18 skeletons.py (moe_routed_kernel: the dispatch
 * contract) and TileOPs-Metax PR #55 (moe_reduce_fused, sections 1-3).
 *
 * Conventions for every entry point:
 *   - Pointers are caller-owned DEVICE memory unless stated otherwise; the
 *     library never allocates device memory.  Inputs are read only; outputs
 *     are fully overwritten (rows/elements the operation defines).
 *   - Tensors are dense, row-major, and 16-byte aligned.  Stacked expert
 *     weights use the nn.Linear (out x in) layout of the pages:
 *     W_gate, W_up [E, d_expert, d_hidden]; W_down [E, d_hidden, d_expert].
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: no host synchronisation and no
 *     device-to-host copy happens inside any call.
 *   - Arguments are validated on the host before anything is launched; a bad
 *     argument returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *     MOE_ERR_WORKSPACE and launches nothing.  A launch failure returns
 *     MOE_ERR_CUDA.  Conditions only the device can see (a combine position
 *     out of range, a pipeline wait that timed out) are written as a non-zero
 *     code into the optional `err_flag` word, which the caller reads after
 *     synchronising; kernels never trap.
 *   - Sizes are int64_t element counts; T = tokens, k = top-k, E = experts,
 *     Tk = T*k token-expert pairs, d_h = d_hidden, d_e = d_expert.
 */
#ifndef MOE_ROUTED_GATE_H
#define MOE_ROUTED_GATE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* identical to cudaStream_t */

/* MOE_E4M3 (float8 e4m3fn) is an output type of moe_reduce_fused_scaled only. */
typedef enum { MOE_F16 = 0, MOE_BF16 = 1, MOE_F32 = 2, MOE_E4M3 = 3 } moe_dtype_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, k > E, misaligned, ... */
    MOE_ERR_UNSUPPORTED = 2, /* a dtype or shape combination the library does not run */
    MOE_ERR_WORKSPACE = 3,   /* workspace smaller than the *_workspace_bytes answer */
    MOE_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
    MOE_ERR_DEVICE_FLAG = 5, /* (err_flag value) a combine position was out of range */
    MOE_ERR_TIMEOUT = 6      /* (err_flag value) a device pipeline wait gave up */
} moe_status_t;

/* Block height of the dispatch padding and of the grouped GEMM tiles. */
#define MOE_BLOCK_M 128

/* Human-readable name of a status code.  Never NULL. */
MOE_API const char *moe_status_string(int status);

/* Number of M blocks of the padded token space: ceil(T*k / block_m) + E
 * (CSDN "forward": M = ceil(B*S*top_k / block_token) + n_routed_experts;
 * skeletons.py moe_routed_kernel: m_blocks).  Returns -1 on bad arguments. */
MOE_API int64_t moe_num_m_blocks(int64_t T, int64_t k, int64_t E, int64_t block_m);

/* Workspace sizes in bytes (0 means none is needed; -1 cast to size_t on bad args). */
MOE_API size_t moe_gate_topk_workspace_bytes(int64_t T, int64_t E);
MOE_API size_t moe_build_dispatch_workspace_bytes(int64_t T, int64_t k, int64_t E);
MOE_API size_t moe_forward_workspace_bytes(int64_t T, int64_t d_h, int64_t d_e, int64_t E, int64_t k,
                                   moe_dtype_t dtype);

/*
 * Gate and routing (CSDN "forward", step 1: expert_indices, expert_scores =
 * gating_network(x); the gate body is not printed on the pages).
 *   logits[t,e] = sum_j x[t,j] * w_g[e,j] (+ bias[e]) in fp32.  The sum order is
 *   fixed: lane L = (j/8) mod 32 accumulates its 8-element chunks in ascending
 *   j with fmaf, then the 32 partials are combined by the xor butterfly
 *   s = 16, 8, 4, 2, 1; this makes the routing reproducible bit for bit.
 *   topk_idx[t, 0..k-1]: the k largest logits, descending, ties to the lower id.
 *   topk_w[t, j] = softmax over all E logits at topk_idx[t, j] (no renormalisation).
 * x [T, d_h] and w_g [E, d_h] in `dtype` (f16 or bf16); bias [E] fp32 or NULL.
 * Requires d_h % 256 == 0, 1 <= k <= min(E, 32), E <= 1024.
 * ws: moe_gate_topk_workspace_bytes(T, E) bytes of scratch, 256-byte aligned;
 * its first T*E*4 bytes receive the fp32 logits [T, E].
 * Many tokens (T >= 1024): the products run on the tensor cores in another
 * summation order, and every expert whose tensor-core logit lies within a
 * stated error bound of the k-th largest is recomputed in the fixed order
 * above, so topk_idx and topk_w are what the fixed order gives (an expert
 * outside the bound cannot be selected).  The logits written then carry the
 * fixed-order value for every recomputed expert (the selected ones among
 * them) and the tensor-core value, within the bound, for the others; the
 * softmax denominator sums those values.  Fewer tokens: every logit is the
 * fixed-order value.
 */
MOE_API moe_status_t moe_gate_topk(const void *x, const void *w_g, const float *bias, int64_t T,
                           int64_t d_h, int64_t E, int64_t k, moe_dtype_t dtype,
                           int32_t *topk_idx, float *topk_w, void *ws, size_t ws_bytes,
                           moe_stream_t stream);

/*
 * Counting-sort dispatch (CSDN "forward", steps 2-5; skeletons.py docstring:
 * the kernel takes four tables and looks up per block which rows it owns).
 *   group_sizes[e]          = #pairs routed to e            (bincount, minlength E)
 *   group_offsets[e]        = exclusive prefix sum of group_sizes
 *   group_padded_offsets[e] = padded start: po[0] = 0,
 *                             po[i] = po[i-1] + ceil((c[i-1] + 1) / block_m) * block_m
 *   group_idx_for_bx[bx]    = last e with bx*block_m >= po[e], bx < moe_num_m_blocks
 *   The pairs f = t*k + j are sorted by expert, stably (ascending f inside an
 *   expert): row r = group_offsets[e] + rank; sorted_token_idx[r] = t,
 *   sorted_row_weight[r] = topk_w[f] (1 when topk_w is NULL),
 *   token_topk_to_pos[f] = r.
 * topk_idx [T,k] int32 with values in [0, E); a pair whose id lies outside
 * that range is dropped (counted nowhere, given no row, its token_topk_to_pos
 * entry left unwritten; nothing is written out of bounds);
 * outputs sized [E], [E], [E], [M_blk], [Tk], [Tk], [Tk].  block_m must be 128.
 * ws: moe_build_dispatch_workspace_bytes(T, k, E) bytes of scratch.
 */
MOE_API moe_status_t moe_build_dispatch(const int32_t *topk_idx, const float *topk_w, int64_t T,
                                int64_t k, int64_t E, int64_t block_m, int32_t *group_sizes,
                                int32_t *group_offsets, int32_t *group_padded_offsets,
                                int32_t *group_idx_for_bx, int32_t *sorted_token_idx,
                                float *sorted_row_weight, int32_t *token_topk_to_pos, void *ws,
                                size_t ws_bytes, moe_stream_t stream);

/*
 * moe_build_dispatch without a workspace argument.  This entry point has no
 * counterpart on the pages; it exists for callers that cannot allocate
 * device memory: code running while a CUDA graph is being captured (where
 * cudaMalloc is not allowed) and engines whose device memory is planned up
 * front by another runtime, so that nothing may be allocated per call.
 * It computes exactly what moe_build_dispatch computes, with the scratch
 * histograms in a fixed 1 MiB array inside the library (every GPU that loads
 * the library holds it until the process exits); it allocates nothing.
 *   - Limit: ceil(T*k / 2048) * E <= 262144 counters (for E = 256 that is up
 *     to 2,097,152 token-expert pairs); larger problems return
 *     MOE_ERR_WORKSPACE without launching.
 *   - Every call made outside a stream capture looks the array's device
 *     address up (cudaGetSymbolAddress, a host-side lookup); a call made
 *     during a capture reuses the address of the last call outside one on
 *     that device.  So make the first call on a device before any stream
 *     capture, and after a cudaDeviceReset (which moves the array) make one
 *     call outside a capture before capturing again.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads) race and give undefined tables.  Nothing needs
 *     clearing between calls: the first kernel writes every counter it reads.
 * Arguments, outputs and errors otherwise as moe_build_dispatch.
 */
MOE_API moe_status_t moe_build_dispatch_noalloc(const int32_t *topk_idx, const float *topk_w,
                                        int64_t T, int64_t k, int64_t E, int64_t block_m,
                                        int32_t *group_sizes, int32_t *group_offsets,
                                        int32_t *group_padded_offsets,
                                        int32_t *group_idx_for_bx, int32_t *sorted_token_idx,
                                        float *sorted_row_weight, int32_t *token_topk_to_pos,
                                        moe_stream_t stream);

/*
 * Stream-ordered copy by a kernel: dst[0, bytes) = src[0, bytes).  Either side
 * may be host memory the device can reach (a pinned allocation's pointer under
 * unified addressing), so a caller can move its tokens in, inside a captured
 * CUDA graph, without a memcpy node (a small copy costs one round trip over
 * the host link; launched with programmatic dependent launch like the
 * forward's kernels).  Not part of the pages' method: plumbing for the
 * forward's end-to-end path.  bytes % 16 == 0, both pointers 16-byte aligned,
 * the ranges must not overlap (MOE_ERR_INVALID_ARG otherwise).
 */
MOE_API moe_status_t moe_copy(const void *src, void *dst, int64_t bytes, moe_stream_t stream);

/*
 * Stream-ordered bounded wait on a flag (a doorbell): work queued after this
 * call on `stream` starts once *flag >= expected, so a pre-launched forward
 * (a replayed CUDA graph, say) can wait for an upstream producer, such as
 * the host filling pinned token buffers or another engine's kernel, without
 * a host synchronisation.  flag: int32 in device memory or in host memory
 * the device can read (a pinned allocation's pointer under unified
 * addressing); it is read with system-scope loads and never written.  Not
 * part of the pages' method: plumbing, like moe_copy.
 * If the flag has not reached `expected` after timeout_ns (1 ns .. 10 s) the
 * wait gives up: *err_flag is set to MOE_ERR_TIMEOUT, the kernel returns and
 * the stream goes on (the CUDA context stays usable; the caller checks
 * *err_flag).  The forward's own kernels bound every wait the same way.
 * err_flag: required device int32.  MOE_ERR_INVALID_ARG for a null pointer
 * or a timeout out of range.
 */
MOE_API moe_status_t moe_wait_flag(const int32_t *flag, int32_t expected, int64_t timeout_ns,
                                   int32_t *err_flag, moe_stream_t stream);

/*
 * Row gather (CSDN "forward", step 3: stacked_expert_tokens[r] = x_flat[token of r]).
 *   a_out[r, :] = x[sorted_token_idx[r], :] for r < n_rows.  x [T, d_h].
 * sorted_token_idx values must lie in [0, T).  d_h * elem_size % 16 == 0.
 */
MOE_API moe_status_t moe_gather_rows(const void *x, const int32_t *sorted_token_idx, int64_t n_rows,
                             int64_t T, int64_t d_h, moe_dtype_t dtype, void *a_out,
                             moe_stream_t stream);

/*
 * The same gather in token order (what moe_forward runs): for every token t
 * and slot j < k, a_out[token_topk_to_pos[t, j], :] = x[t, :]; a position
 * outside [0, n_rows) (a dropped pair, -1) is skipped and rows no position
 * names are left as they were.  With a dispatch's token_topk_to_pos (every
 * row named exactly once) the result is moe_gather_rows' with that
 * dispatch's sorted_token_idx, but each token's row is read from memory once
 * instead of once per expert it went to.  token_topk_to_pos [T, k] int32,
 * 1 <= k <= 32.  x [T, d_h]; d_h * elem_size % 16 == 0.  The rows move by
 * bulk copies through shared memory (one load per token, one store per
 * row); err_flag: optional device int32, set to MOE_ERR_TIMEOUT if a copy
 * wait gives up (the rows of the token that timed out and of the tokens
 * after it in its stream are then not written).
 */
MOE_API moe_status_t moe_gather_rows_by_token(const void *x, const int32_t *token_topk_to_pos, int64_t T,
                                              int64_t k, int64_t n_rows, int64_t d_h, moe_dtype_t dtype,
                                              void *a_out, int32_t *err_flag, moe_stream_t stream);

/*
 * Grouped gate/up GEMM with fused SiLU (CSDN "tilelang kernel stage 1 gate+up";
 * skeletons.py moe_routed_kernel first kernel).  For each M block bx:
 *   g = group_idx_for_bx[bx]; m_start = bx*128 - group_padded_offsets[g] + group_offsets[g];
 *   rows = clamp(group_sizes[g] - (bx*128 - group_padded_offsets[g]), 0, 128);
 *   h[m_start + i, :] = silu(A_i W_gate[g]^T) * (A_i W_up[g]^T), i < rows,
 * fp32 accumulation on the tensor cores, rounded once to `dtype`.
 * a [n_rows, d_h]; w_gate, w_up [E, d_e, d_h]; h [n_rows, d_e]; tables as produced
 * by moe_build_dispatch for (T, k) with T*k == n_rows.  dtype f16 or bf16;
 * d_h % 64 == 0, d_e % 64 == 0.  Rows of h outside the tables' rows are not written.
 * err_flag: optional device int32, set to MOE_ERR_TIMEOUT if a pipeline wait gives up.
 */
MOE_API moe_status_t moe_grouped_gate_up_silu(const void *a, const void *w_gate, const void *w_up,
                                      const int32_t *group_sizes, const int32_t *group_offsets,
                                      const int32_t *group_padded_offsets,
                                      const int32_t *group_idx_for_bx, int64_t m_blocks,
                                      int64_t n_rows, int64_t d_h, int64_t d_e, int64_t E,
                                      moe_dtype_t dtype, void *h, int32_t *err_flag,
                                      moe_stream_t stream);

/*
 * Grouped down GEMM (CSDN "tilelang kernel stage 2 down"; skeletons.py second
 * kernel).  Same block lookup; y[m_start + i, :] = (h_i W_down[g]^T) * rw_i,
 * rw_i = row_weights[m_start + i] when row_weights is non-NULL, else 1 (the
 * forward applies the routing weight once, in the combine).  fp32 accumulation,
 * rounded once to `dtype`.  h [n_rows, d_e]; w_down [E, d_h, d_e]; y [n_rows, d_h].
 * d_h % 256 == 0, d_e % 64 == 0.
 */
MOE_API moe_status_t moe_grouped_down(const void *h, const void *w_down, const int32_t *group_sizes,
                              const int32_t *group_offsets, const int32_t *group_padded_offsets,
                              const int32_t *group_idx_for_bx, int64_t m_blocks,
                              const float *row_weights, int64_t n_rows, int64_t d_h,
                              int64_t d_e, int64_t E, moe_dtype_t dtype, void *y,
                              int32_t *err_flag, moe_stream_t stream);

/*
 * Both expert GEMMs in one persistent launch (CSDN "tilelang kernel stage 2
 * down": the article names fusing the two stages as an optimisation point).
 * Results equal moe_grouped_gate_up_silu(a -> h) followed by
 * moe_grouped_down(h -> y, row_weights): h [n_rows, d_e] is still written (it
 * is stage 2's operand, read back mostly from L2) and y [n_rows, d_h].
 * Inside the kernel a stage-2 tile starts once all stage-1 tiles of its M
 * block are stored, and each CTA takes its next tile from a shared counter.
 * `ready` is caller-owned device memory of m_blocks + 1 int32 (the per-block
 * counters, then the tile counter) that this call zeroes (stream ordered)
 * before the launch.
 * Gathering form: with sorted_token_idx non-NULL, stage 1 reads its rows from
 * the tokens x [T, d_h] by those indices (the gather of the CSDN "forward",
 * step 3, done by four-row TMA gathers in the kernel) and `a` is not read;
 * T >= 1 is the number of rows of x (every index must be below it).  It pays
 * when blocks are small (at most 64 rows); a full 128-row tile is read faster
 * from gathered rows `a`.  Otherwise x and T are ignored and may be NULL / 0.
 * Every tile is taken from the shared counter in order, and all stage-1
 * tiles come before all stage-2 tiles, so a stage-2 tile only waits on tiles
 * that running CTAs hold: the launch completes whether or not all its CTAs
 * (one per SM) are resident at once.  The waits are bounded all the same:
 * after about 2 s *err_flag is set to MOE_ERR_TIMEOUT and the kernel
 * returns.  Other arguments, layouts and errors as the two calls.
 */
MOE_API moe_status_t moe_grouped_mlp(const void *a, const void *w_gate, const void *w_up,
                             const void *w_down, const int32_t *group_sizes,
                             const int32_t *group_offsets, const int32_t *group_padded_offsets,
                             const int32_t *group_idx_for_bx, int64_t m_blocks,
                             const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                             int64_t E, moe_dtype_t dtype, void *h, void *y, int32_t *ready,
                             const void *x, const int32_t *sorted_token_idx, int64_t T,
                             int32_t *err_flag, moe_stream_t stream);

/*
 * Weight-only int4 experts (W4A16; TileLang tutorial ch.18 skeletons.py,
 * w4a8_dequant_gemm and its notes on quantisation: int4 weights two per
 * byte, element j of a row in byte j/2 at nibble j%2 from the low end, two's
 * complement, unpacked on chip and cast to the 16-bit compute type).
 *
 * moe_pack_int4_bytes / moe_pack_int4_weights: a stacked weight [E, N, K]
 * in that format (plain: E*N*K/2 bytes) rewritten into the tiled layout the
 * int4 kernels read: tiles of tile_rows output channels (128 for W_gate and
 * W_up, N = d_e, K = d_h; 256 for W_down, N = d_h, K = d_e), stored
 * [E][ceil(N/tile_rows)][K/64][tile_rows][32 bytes] so that one 64-wide K
 * step of a tile is one contiguous block; inside each 4-byte word elements
 * 2m, 2m+1 sit in nibbles m, m+4 as value + 8; rows past N hold zeros.
 * moe_pack_int4_bytes returns the packed size (-1 for K % 64 != 0, sizes
 * <= 0 or another tile_rows).  Device pointers, 16-byte aligned, distinct.
 * Done once when the weights are loaded.
 */
MOE_API int64_t moe_pack_int4_bytes(int64_t E, int64_t N, int64_t K, int64_t tile_rows);
MOE_API moe_status_t moe_pack_int4_weights(const uint8_t *plain, int64_t E, int64_t N, int64_t K,
                                   int64_t tile_rows, uint8_t *packed, moe_stream_t stream);

/*
 * Both expert stages in one launch with int4 weights, for any T >= 1
 * (the kernel works on units of at most 64 rows: a 128-row block of the
 * tables with more rows is two units; it is built for decode-sized T,
 * where the weight bytes are the cost, and unpacks each weight tile once
 * per unit, so large T is correct but slow):
 *   stage 1: G = (A q_gate[g]^T) * s_gate[g], U = (A q_up[g]^T) * s_up[g],
 *            h = rt(silu(G) * U)       (A: rows of x gathered by sorted_token_idx)
 *   stage 2: y = rt((h q_down[g]^T) * s_down[g] (* row_weights))
 * in fp32 accumulators; q_* are moe_pack_int4_weights output (q_gate, q_up
 * with tile_rows 128, q_down with 256); s_* fp32 per output channel
 * ([E, d_e], [E, d_e], [E, d_h]) or NULL for 1 (the pages print no scale;
 * reading: a per-channel scale on the fp32 sum).  x [T, d_h] in `dtype`;
 * h [n_rows, d_e], y [n_rows, d_h]; ready as moe_grouped_mlp (m_blocks + 1
 * int32, zeroed by this call).  d_h % 64 == 0, d_e % 64 == 0,
 * m_blocks <= 1088 (else MOE_ERR_UNSUPPORTED).  Waits bounded as
 * moe_grouped_mlp.
 */
MOE_API moe_status_t moe_grouped_mlp_w4a16(const void *x, const int32_t *sorted_token_idx, int64_t T,
                                   const uint8_t *q_gate, const uint8_t *q_up, const uint8_t *q_down,
                                   const float *s_gate, const float *s_up, const float *s_down,
                                   const int32_t *group_sizes, const int32_t *group_offsets,
                                   const int32_t *group_padded_offsets,
                                   const int32_t *group_idx_for_bx, int64_t m_blocks,
                                   const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                                   int64_t E, moe_dtype_t dtype, void *h, void *y, int32_t *ready,
                                   int32_t *err_flag, moe_stream_t stream);

/*
 * W4A8: int4 weights times int8 activations, summed exactly into int32
 * (TileLang tutorial ch.18 skeletons.py, w4a8_dequant_gemm: the packed int4
 * weight is unpacked and sign-extended on chip, the products summed in an
 * int32 accumulator, the result written transposed; the module notes on
 * quantisation: weight + activation quantisation, W4A8).  The results are
 * the exact integer sums (bit-identical to an integer GEMM); the skeleton
 * applies no scale, so none is taken here.
 *
 * moe_gemm_w4a8: Ct[n, m] = sum_k A[m, k] * int4(B)[n, k].  A int8 [M, K]
 * row-major; B the weight [N, K] in the int4 format, packed by
 * moe_pack_int4_weights with E = 1 and tile_rows = 256; Ct int32 [N, M]
 * (transposed, as the skeleton writes it).  1 <= M <= 64 (the decode and
 * small-batch shapes; M > 64 is MOE_ERR_UNSUPPORTED), N >= 1, K % 64 == 0,
 * 64 <= K <= 2^20 (|Ct| <= 1024 K cannot overflow int32).  ws: device
 * scratch of moe_gemm_w4a8_workspace_bytes(M, K) bytes (-1 for bad sizes),
 * owned by the caller, 16-byte aligned, used only by this call's work (for
 * M <= 8 the call streams the weights through the CUDA cores, dp4a on the
 * packed bytes, and leaves ws untouched; larger M use the tensor cores).
 * A, B, ws 16-byte aligned, Ct 4-byte aligned, all distinct.
 *
 * moe_grouped_gemm_w4a8: the same per routed row over the dispatch tables
 * (the block walk of moe_routed_kernel): C[r, n] = sum_k x[i_r, k] *
 * int4(B[g])[n, k] with g the expert of row r and i_r = sorted_token_idx[r]
 * (NULL: i_r = r, n_rows <= T).  x int8 [T, K], T >= 1 (64-row units as
 * moe_grouped_mlp_w4a16), B [E, N, K] packed with tile_rows 256,
 * C int32 [n_rows, N].  A sorted_token_idx entry outside [0, T) is reported
 * on err_flag (MOE_ERR_DEVICE_FLAG) and its row of C summed from zeros.
 * ws: moe_grouped_gemm_w4a8_workspace_bytes(n_rows, K, m_blocks) bytes.
 * m_blocks <= 1088.  Waits bounded as moe_grouped_mlp.
 */
MOE_API int64_t moe_gemm_w4a8_workspace_bytes(int64_t M, int64_t K);
MOE_API moe_status_t moe_gemm_w4a8(const int8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K,
                                   int32_t *Ct, void *ws, int64_t ws_bytes, int32_t *err_flag,
                                   moe_stream_t stream);
MOE_API int64_t moe_grouped_gemm_w4a8_workspace_bytes(int64_t n_rows, int64_t K, int64_t m_blocks);
MOE_API moe_status_t moe_grouped_gemm_w4a8(const int8_t *x, const int32_t *sorted_token_idx, int64_t T,
                                           const uint8_t *B, const int32_t *group_sizes,
                                           const int32_t *group_offsets, const int32_t *group_padded_offsets,
                                           const int32_t *group_idx_for_bx, int64_t m_blocks, int64_t n_rows,
                                           int64_t N, int64_t K, int64_t E, int32_t *C, void *ws,
                                           int64_t ws_bytes, int32_t *err_flag, moe_stream_t stream);

/*
 * moe_reduce_fused (TileOPs-Metax PR #55, section 1): for every token t and
 * hidden element h,
 *   out[t, h] = cast( sum over k ascending with 0 <= pos[t,k] < n_rows of
 *                     w[t,k] * x[pos[t,k], h] )
 * accumulated in fp32 as acc = acc + (w * x) starting from +0, cast once.
 * pos = token_topk_to_pos [T, K] int32, -1 marks a padding slot (skipped);
 * w = topk_weights [T, K] fp32, or NULL for unit weights.  x [n_rows, H].
 * Requires H % 256 == 0 (the page's check).  Dtypes: in == out (f16, bf16,
 * f32), or f32 in with f16/bf16 out.  A pos < -1 or >= n_rows is skipped and
 * sets *err_flag = MOE_ERR_DEVICE_FLAG when err_flag is non-NULL.
 */
MOE_API moe_status_t moe_reduce_fused(const void *x, int64_t n_rows, const int32_t *token_topk_to_pos,
                              const float *topk_weights, int64_t T, int64_t K, int64_t H,
                              moe_dtype_t in_dtype, moe_dtype_t out_dtype, void *out,
                              int32_t *err_flag, moe_stream_t stream);

/*
 * moe_reduce_fused with the scaling and output switches of TileOPs-Metax
 * PR #55's op variants (WithXsf, Fp8, Quantized; section 1 "variants inlined
 * into one kernel", commit "correct roofline FLOPs for the scaling variants"):
 *   s[t,k]   = w[t,k] * x_sf[pos[t,k]]     x_sf: one fp32 scale per row of x
 *                                            (per routed slot), or NULL = 1
 *   acc[t,h] = sum over k ascending, valid pos, of s[t,k] * x[pos[t,k], h]
 *   out[t,h] = cast(acc[t,h] * sf[t])        sf: one fp32 scale per token, or NULL
 * with the same fp32 order and roundings as moe_reduce_fused (each product
 * and sum rounded; sf applied after the sum).  out_dtype may be MOE_E4M3:
 * float8 e4m3fn, round to nearest even, finite values saturated to +-448.
 * x_sf has n_rows entries, sf has T.  Other arguments and errors as
 * moe_reduce_fused.
 */
MOE_API moe_status_t moe_reduce_fused_scaled(const void *x, int64_t n_rows,
                                     const int32_t *token_topk_to_pos, const float *topk_weights,
                                     const float *x_sf, const float *sf, int64_t T, int64_t K,
                                     int64_t H, moe_dtype_t in_dtype, moe_dtype_t out_dtype,
                                     void *out, int32_t *err_flag, moe_stream_t stream);

/*
 * The whole routed forward (CSDN "tilelang baseline": the custom_kernel entry
 * that takes the tokens, the gate and the stacked expert weights and returns
 * the layer output, and the "forward" section that composes routing, the
 * table build, the two expert kernels and the weighted combine), stream
 * ordered, no host round trip:
 *   moe_gate_topk -> moe_build_dispatch -> moe_gather_rows_by_token ->
 *   moe_grouped_mlp (stage 1 + stage 2 in one launch) -> moe_reduce_fused;
 * for T <= 64 the gather is done inside moe_grouped_mlp (its gathering form)
 * and the gathered-rows section of the workspace is left unwritten.
 * x [T, d_h]; w_g [E, d_h]; bias [E] fp32 or NULL; w_gate/w_up [E, d_e, d_h];
 * w_down [E, d_h, d_e]; out [T, d_h]; all in `dtype` (f16 or bf16).  `out`
 * may also be host memory the device can store to (a pinned allocation's
 * pointer under unified addressing): the combine writes it with plain
 * stores, so the result reaches the host without a separate copy.
 * ws: moe_forward_workspace_bytes(...) bytes, 256-byte aligned; it holds every
 * intermediate (routing, tables, gathered rows, h, y) and is not read before
 * being written, so it needs no clearing.  err_flag: optional device int32.
 */
MOE_API moe_status_t moe_forward(const void *x, const void *w_g, const float *bias, const void *w_gate,
                         const void *w_up, const void *w_down, int64_t T, int64_t d_h,
                         int64_t d_e, int64_t E, int64_t k, moe_dtype_t dtype, void *ws,
                         size_t ws_bytes, void *out, int32_t *err_flag, moe_stream_t stream);

/*
 * moe_forward with int4 experts (moe_grouped_mlp_w4a16 as the expert MLP,
 * which gathers its rows from x), for T >= 1 tokens with at most 1088
 * M blocks (else MOE_ERR_UNSUPPORTED); the gate weight w_g stays in
 * `dtype`.  Same workspace (moe_forward_workspace_bytes) and outputs as
 * moe_forward.
 */
MOE_API moe_status_t moe_forward_w4a16(const void *x, const void *w_g, const float *bias,
                               const uint8_t *q_gate, const uint8_t *q_up, const uint8_t *q_down,
                               const float *s_gate, const float *s_up, const float *s_down,
                               int64_t T, int64_t d_h, int64_t d_e, int64_t E, int64_t k,
                               moe_dtype_t dtype, void *ws, size_t ws_bytes, void *out,
                               int32_t *err_flag, moe_stream_t stream);

/*
 * Offsets (bytes from the workspace start) of moe_forward's intermediates, for
 * inspection after a call: index 0 logits, 1 topk_idx, 2 topk_w, 3 group_sizes,
 * 4 group_offsets, 5 group_padded_offsets, 6 group_idx_for_bx,
 * 7 sorted_token_idx, 8 sorted_row_weight, 9 token_topk_to_pos, 10 dispatch
 * scratch, 11 gathered rows A, 12 h, 13 y, 14 the per-block counters of
 * moe_grouped_mlp.  Returns -1 for a bad index.
 */
MOE_API int64_t moe_forward_workspace_offset(int64_t T, int64_t d_h, int64_t d_e, int64_t E, int64_t k,
                                     moe_dtype_t dtype, int index);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTED_GATE_H */

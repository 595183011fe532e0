// capi.cu -- the exported C-ABI: host-side argument checks, workspace layout,
// and the stream-ordered composition of the forward.  See the public header
// for the contract of every entry point.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>

#include "../../include/moe_routed_gate.h"
#include "internal.h"

namespace moe {

int device_sm_count() {
    static std::atomic<int> cached[64];  // zero-initialised; several host threads may call
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 152;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    if (dev < 64) cached[dev] = n;
    return n;
}

int mlp_grid(int64_t tiles) {
    // MOE_MLP_GRID: a CTA count for the persistent expert-MLP launches in place
    // of one CTA per SM (read at every launch; tests use it to run the kernel
    // on fewer CTAs, or on more CTAs than fit on the GPU at once)
    int64_t grid = device_sm_count();
    if (const char *v = std::getenv("MOE_MLP_GRID")) {
        const long n = std::strtol(v, nullptr, 10);
        if (n >= 1 && n <= 65535) grid = n;
    }
    return static_cast<int>(tiles < grid ? tiles : grid);
}

bool mlp_pairs_enabled() {
    // MOE_MLP_PAIRS=0 keeps the expert MLP on the one-SM kernel (tests compare
    // the two forms); read at every launch
    const char *v = std::getenv("MOE_MLP_PAIRS");
    return !(v && v[0] == '0');
}

}  // namespace moe

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_half_type(moe_dtype_t d) { return d == MOE_F16 || d == MOE_BF16; }

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int64_t m_blocks_of(int64_t T, int64_t k, int64_t E, int64_t block_m) {
    if (T < 0 || k <= 0 || E <= 0 || block_m <= 0) return -1;
    return (T * k + block_m - 1) / block_m + E;
}

constexpr int kFwdSections = 15;

struct FwdLayout {
    size_t off[kFwdSections];
    size_t total;
};

bool fwd_layout(int64_t T, int64_t d_h, int64_t d_e, int64_t E, int64_t k, moe_dtype_t dtype,
                FwdLayout *L) {
    if (T < 0 || d_h <= 0 || d_e <= 0 || E <= 0 || k <= 0 || !is_half_type(dtype)) return false;
    const size_t es = 2;
    const size_t Tk = static_cast<size_t>(T * k);
    const size_t mb = static_cast<size_t>(m_blocks_of(T, k, E, MOE_BLOCK_M));
    const size_t sz[kFwdSections] = {
        moe_gate_topk_workspace_bytes(T, E),  // 0 logits (+ the tensor-core gate's scratch)
        Tk * 4,                          // 1 topk_idx
        Tk * 4,                          // 2 topk_w
        static_cast<size_t>(E) * 4,      // 3 group_sizes
        static_cast<size_t>(E) * 4,      // 4 group_offsets
        static_cast<size_t>(E) * 4,      // 5 group_padded_offsets
        mb * 4,                          // 6 group_idx_for_bx
        Tk * 4,                          // 7 sorted_token_idx
        Tk * 4,                          // 8 sorted_row_weight
        Tk * 4,                          // 9 token_topk_to_pos
        moe::dispatch_scratch_bytes(static_cast<int64_t>(Tk), E),  // 10 dispatch scratch
        Tk * d_h * es,                   // 11 A (gathered rows)
        Tk * d_e * es,                   // 12 h
        Tk * d_h * es,                   // 13 y
        (mb + 1) * 4,                    // 14 per-block counters + tile counter of the expert MLP
    };
    size_t cur = 0;
    for (int i = 0; i < kFwdSections; ++i) {
        L->off[i] = cur;
        cur += align_up(sz[i] > 0 ? sz[i] : 1);
    }
    L->total = cur;
    return true;
}

}  // namespace

extern "C" {

const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: unsupported dtype or shape";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
        case MOE_ERR_DEVICE_FLAG: return "MOE_ERR_DEVICE_FLAG: out-of-range position seen on the device";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a device pipeline wait timed out";
        default: return "unknown moe status";
    }
}

int64_t moe_num_m_blocks(int64_t T, int64_t k, int64_t E, int64_t block_m) {
    return m_blocks_of(T, k, E, block_m);
}

size_t moe_gate_topk_workspace_bytes(int64_t T, int64_t E) {
    if (T < 0 || E <= 0) return static_cast<size_t>(-1);
    return align_up(static_cast<size_t>(T) * static_cast<size_t>(E) * 4) + moe::gate_tc_scratch_bytes(T, E);
}

size_t moe_build_dispatch_workspace_bytes(int64_t T, int64_t k, int64_t E) {
    if (T < 0 || k <= 0 || E <= 0) return static_cast<size_t>(-1);
    return moe::dispatch_scratch_bytes(T * k, E);
}

size_t moe_forward_workspace_bytes(int64_t T, int64_t d_h, int64_t d_e, int64_t E, int64_t k,
                                   moe_dtype_t dtype) {
    FwdLayout L;
    if (!fwd_layout(T, d_h, d_e, E, k, dtype, &L)) return static_cast<size_t>(-1);
    return L.total;
}

int64_t moe_forward_workspace_offset(int64_t T, int64_t d_h, int64_t d_e, int64_t E, int64_t k,
                                     moe_dtype_t dtype, int index) {
    FwdLayout L;
    if (index < 0 || index >= kFwdSections || !fwd_layout(T, d_h, d_e, E, k, dtype, &L)) return -1;
    return static_cast<int64_t>(L.off[index]);
}

static moe_status_t gate_topk(const void *x, const void *w_g, const float *bias, int64_t T,
                              int64_t d_h, int64_t E, int64_t k, moe_dtype_t dtype,
                              int32_t *topk_idx, float *topk_w, void *ws, size_t ws_bytes,
                              int32_t *err_flag, moe_stream_t stream) {
    if (T < 0 || d_h <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (d_h % 256 != 0 || k > E || k > 32 || E > 1024) return MOE_ERR_INVALID_ARG;
    if (!is_half_type(dtype)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !w_g || !topk_idx || !topk_w || !ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_g) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0)
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_gate_topk_workspace_bytes(T, E)) return MOE_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float *logits = static_cast<float *>(ws);
    // the tensor-core gate's scratch follows the logits (present for many tokens)
    void *tc_scratch = moe::gate_tc_scratch_bytes(T, E) > 0
                           ? static_cast<char *>(ws) + align_up(static_cast<size_t>(T) * E * 4)
                           : nullptr;
    return cuda_status(moe::launch_gate_topk(x, w_g, bias, T, d_h, E, k, dtype, logits, topk_idx,
                                             topk_w, tc_scratch, err_flag, s));
}

moe_status_t moe_gate_topk(const void *x, const void *w_g, const float *bias, int64_t T,
                           int64_t d_h, int64_t E, int64_t k, moe_dtype_t dtype,
                           int32_t *topk_idx, float *topk_w, void *ws, size_t ws_bytes,
                           moe_stream_t stream) {
    return gate_topk(x, w_g, bias, T, d_h, E, k, dtype, topk_idx, topk_w, ws, ws_bytes, nullptr,
                     stream);
}

}  // extern "C"

namespace moe {

int check_dispatch_args(const int32_t *topk_idx, int64_t T, int64_t k, int64_t E, int64_t block_m,
                        const int32_t *group_sizes, const int32_t *group_offsets,
                        const int32_t *group_padded_offsets, const int32_t *group_idx_for_bx,
                        const int32_t *sorted_token_idx, const float *sorted_row_weight,
                        const int32_t *token_topk_to_pos) {
    if (T < 0 || k <= 0 || E <= 0 || E > 1024 || block_m != MOE_BLOCK_M) return MOE_ERR_INVALID_ARG;
    if (T * k > (int64_t(1) << 30)) return MOE_ERR_UNSUPPORTED;
    if (!group_sizes || !group_offsets || !group_padded_offsets || !group_idx_for_bx)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !sorted_token_idx || !sorted_row_weight || !token_topk_to_pos))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace moe

extern "C" {

static moe_status_t build_dispatch(const int32_t *topk_idx, const float *topk_w, int64_t T,
                                   int64_t k, int64_t E, int64_t block_m, int32_t *group_sizes,
                                   int32_t *group_offsets, int32_t *group_padded_offsets,
                                   int32_t *group_idx_for_bx, int32_t *sorted_token_idx,
                                   float *sorted_row_weight, int32_t *token_topk_to_pos, void *ws,
                                   size_t ws_bytes, int32_t *ready, moe_stream_t stream) {
    const int st = moe::check_dispatch_args(topk_idx, T, k, E, block_m, group_sizes, group_offsets,
                                            group_padded_offsets, group_idx_for_bx,
                                            sorted_token_idx, sorted_row_weight, token_topk_to_pos);
    if (st != MOE_OK) return static_cast<moe_status_t>(st);
    const size_t need = moe_build_dispatch_workspace_bytes(T, k, E);
    if (T > 0 && (ws_bytes < need || !ws)) return MOE_ERR_WORKSPACE;
    return cuda_status(moe::launch_dispatch(
        topk_idx, topk_w, T, k, E, block_m, group_sizes, group_offsets, group_padded_offsets,
        group_idx_for_bx, m_blocks_of(T, k, E, block_m), sorted_token_idx, sorted_row_weight,
        token_topk_to_pos, ws, ready, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_build_dispatch(const int32_t *topk_idx, const float *topk_w, int64_t T,
                                int64_t k, int64_t E, int64_t block_m, int32_t *group_sizes,
                                int32_t *group_offsets, int32_t *group_padded_offsets,
                                int32_t *group_idx_for_bx, int32_t *sorted_token_idx,
                                float *sorted_row_weight, int32_t *token_topk_to_pos, void *ws,
                                size_t ws_bytes, moe_stream_t stream) {
    return build_dispatch(topk_idx, topk_w, T, k, E, block_m, group_sizes, group_offsets,
                          group_padded_offsets, group_idx_for_bx, sorted_token_idx,
                          sorted_row_weight, token_topk_to_pos, ws, ws_bytes, nullptr, stream);
}

moe_status_t moe_gather_rows(const void *x, const int32_t *sorted_token_idx, int64_t n_rows,
                             int64_t T, int64_t d_h, moe_dtype_t dtype, void *a_out,
                             moe_stream_t stream) {
    if (n_rows < 0 || T < 0 || d_h <= 0) return MOE_ERR_INVALID_ARG;
    const int es = dtype == MOE_F32 ? 4 : 2;
    if (dtype != MOE_F16 && dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
    if ((d_h * es) % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0) return MOE_OK;
    if (!x || !sorted_token_idx || !a_out || !aligned16(x) || !aligned16(a_out))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_gather_rows(x, sorted_token_idx, n_rows, d_h, es, a_out,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_gather_rows_by_token(const void *x, const int32_t *token_topk_to_pos, int64_t T, int64_t k,
                                      int64_t n_rows, int64_t d_h, moe_dtype_t dtype, void *a_out,
                                      int32_t *err_flag, moe_stream_t stream) {
    if (n_rows < 0 || T < 0 || d_h <= 0 || k <= 0 || k > 32) return MOE_ERR_INVALID_ARG;
    const int es = dtype == MOE_F32 ? 4 : 2;
    if (dtype != MOE_F16 && dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
    if ((d_h * es) % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0 || T == 0) return MOE_OK;
    if (!x || !token_topk_to_pos || !a_out || !aligned16(x) || !aligned16(a_out)) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_scatter_rows(x, token_topk_to_pos, T, k, n_rows, d_h, es, a_out, err_flag,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_copy(const void *src, void *dst, int64_t bytes, moe_stream_t stream) {
    if (bytes < 0 || bytes % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (bytes == 0) return MOE_OK;
    if (!src || !dst || !aligned16(src) || !aligned16(dst)) return MOE_ERR_INVALID_ARG;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
    if (s0 < d0 + static_cast<uintptr_t>(bytes) && d0 < s0 + static_cast<uintptr_t>(bytes))
        return MOE_ERR_INVALID_ARG;  // overlapping
    return cuda_status(moe::launch_copy(src, dst, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_wait_flag(const int32_t *flag, int32_t expected, int64_t timeout_ns, int32_t *err_flag,
                           moe_stream_t stream) {
    if (!flag || !err_flag || timeout_ns < 1 || timeout_ns > 10000000000ll) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_wait_flag(flag, expected, timeout_ns, err_flag,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

static moe_status_t check_gemm_tables(const int32_t *s, const int32_t *o, const int32_t *p,
                                      const int32_t *g, int64_t m_blocks, int64_t n_rows, int64_t E) {
    if (!s || !o || !p || !g) return MOE_ERR_INVALID_ARG;
    if (m_blocks <= 0 || n_rows <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
    if (m_blocks > (n_rows + MOE_BLOCK_M - 1) / MOE_BLOCK_M + E) return MOE_ERR_INVALID_ARG;
    if (n_rows > (int64_t(1) << 31) - 256) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status_t moe_grouped_gate_up_silu(const void *a, const void *w_gate, const void *w_up,
                                      const int32_t *group_sizes, const int32_t *group_offsets,
                                      const int32_t *group_padded_offsets,
                                      const int32_t *group_idx_for_bx, int64_t m_blocks,
                                      int64_t n_rows, int64_t d_h, int64_t d_e, int64_t E,
                                      moe_dtype_t dtype, void *h, int32_t *err_flag,
                                      moe_stream_t stream) {
    if (!is_half_type(dtype)) return MOE_ERR_UNSUPPORTED;
    if (d_h <= 0 || d_e <= 0 || d_h % 64 != 0 || d_e % 64 != 0) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0) return MOE_OK;
    moe_status_t st = check_gemm_tables(group_sizes, group_offsets, group_padded_offsets,
                                        group_idx_for_bx, m_blocks, n_rows, E);
    if (st != MOE_OK) return st;
    if (!a || !w_gate || !w_up || !h) return MOE_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(h))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_grouped_gemm(
        true, dtype, a, w_gate, w_up, group_sizes, group_offsets, group_padded_offsets,
        group_idx_for_bx, m_blocks, nullptr, n_rows, d_h, d_e, E, h, err_flag,
        reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_grouped_down(const void *h, const void *w_down, const int32_t *group_sizes,
                              const int32_t *group_offsets, const int32_t *group_padded_offsets,
                              const int32_t *group_idx_for_bx, int64_t m_blocks,
                              const float *row_weights, int64_t n_rows, int64_t d_h,
                              int64_t d_e, int64_t E, moe_dtype_t dtype, void *y,
                              int32_t *err_flag, moe_stream_t stream) {
    if (!is_half_type(dtype)) return MOE_ERR_UNSUPPORTED;
    if (d_h <= 0 || d_e <= 0 || d_h % 64 != 0 || d_e % 64 != 0) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0) return MOE_OK;
    moe_status_t st = check_gemm_tables(group_sizes, group_offsets, group_padded_offsets,
                                        group_idx_for_bx, m_blocks, n_rows, E);
    if (st != MOE_OK) return st;
    if (!h || !w_down || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(w_down) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_grouped_gemm(
        false, dtype, h, w_down, nullptr, group_sizes, group_offsets, group_padded_offsets,
        group_idx_for_bx, m_blocks, row_weights, n_rows, d_e, d_h, E, y, err_flag,
        reinterpret_cast<cudaStream_t>(stream)));
}

// zero_ready: clear the counters on the stream first (the forward has its
// dispatch kernel clear them instead, keeping the kernels back to back).
// gather_idx: stage 1 gathers token rows of x [T, d_h] by these indices
// instead of reading `a`.
static moe_status_t grouped_mlp(const void *a, const void *w_gate, const void *w_up,
                                const void *w_down, const int32_t *group_sizes,
                                const int32_t *group_offsets, const int32_t *group_padded_offsets,
                                const int32_t *group_idx_for_bx, int64_t m_blocks,
                                const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                                int64_t E, moe_dtype_t dtype, void *h, void *y, int32_t *ready,
                                int32_t *err_flag, moe_stream_t stream, bool zero_ready,
                                const void *x = nullptr, const int32_t *gather_idx = nullptr,
                                int64_t T = 0) {
    if (!is_half_type(dtype)) return MOE_ERR_UNSUPPORTED;
    if (d_h <= 0 || d_e <= 0 || d_h % 64 != 0 || d_e % 64 != 0) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0) return MOE_OK;
    moe_status_t st = check_gemm_tables(group_sizes, group_offsets, group_padded_offsets,
                                        group_idx_for_bx, m_blocks, n_rows, E);
    if (st != MOE_OK) return st;
    const void *rows_in = gather_idx ? x : a;
    if (!rows_in || !w_gate || !w_up || !w_down || !h || !y || !ready) return MOE_ERR_INVALID_ARG;
    if (gather_idx && (T <= 0 || T > INT32_MAX)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(rows_in) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(h) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (zero_ready) {
        cudaError_t e = cudaMemsetAsync(ready, 0, static_cast<size_t>(m_blocks + 1) * 4, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    // many rows, pre-gathered, no row weight: both stages on pairs of SMs
    if (!gather_idx && !row_weights && moe::mlp_pairs_enabled() &&
        moe::grouped_mlp2_applies(n_rows, d_h, d_e, E))
        return cuda_status(moe::launch_grouped_mlp2(dtype, a, w_gate, w_up, w_down, group_sizes,
                                                    group_offsets, group_padded_offsets, m_blocks, n_rows,
                                                    d_h, d_e, E, h, y, ready, err_flag, s));
    return cuda_status(moe::launch_grouped_mlp(dtype, a, w_gate, w_up, w_down, group_sizes,
                                               group_offsets, group_padded_offsets, group_idx_for_bx,
                                               m_blocks, row_weights, n_rows, d_h, d_e, E, h, y,
                                               ready, err_flag, s, x, gather_idx, T));
}

moe_status_t moe_grouped_mlp(const void *a, const void *w_gate, const void *w_up,
                             const void *w_down, const int32_t *group_sizes,
                             const int32_t *group_offsets, const int32_t *group_padded_offsets,
                             const int32_t *group_idx_for_bx, int64_t m_blocks,
                             const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                             int64_t E, moe_dtype_t dtype, void *h, void *y, int32_t *ready,
                             const void *x, const int32_t *sorted_token_idx, int64_t T,
                             int32_t *err_flag, moe_stream_t stream) {
    return grouped_mlp(a, w_gate, w_up, w_down, group_sizes, group_offsets, group_padded_offsets,
                       group_idx_for_bx, m_blocks, row_weights, n_rows, d_h, d_e, E, dtype, h, y,
                       ready, err_flag, stream, true, x, sorted_token_idx, T);
}

int64_t moe_pack_int4_bytes(int64_t E, int64_t N, int64_t K, int64_t tile_rows) {
    if (tile_rows != 128 && tile_rows != 256) return -1;
    return moe::pack_int4_bytes(E, N, K, static_cast<int>(tile_rows));
}

moe_status_t moe_pack_int4_weights(const uint8_t *plain, int64_t E, int64_t N, int64_t K,
                                   int64_t tile_rows, uint8_t *packed, moe_stream_t stream) {
    if (moe_pack_int4_bytes(E, N, K, tile_rows) < 0) return MOE_ERR_INVALID_ARG;
    if (!plain || !packed || plain == packed || !aligned16(plain) || !aligned16(packed))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_pack_int4(plain, E, N, K, static_cast<int>(tile_rows), packed,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

// zero_ready as in grouped_mlp
static moe_status_t grouped_mlp_w4(const void *x, const int32_t *sorted_token_idx, int64_t T,
                                   const uint8_t *q_gate, const uint8_t *q_up, const uint8_t *q_down,
                                   const float *s_gate, const float *s_up, const float *s_down,
                                   const int32_t *group_sizes, const int32_t *group_offsets,
                                   const int32_t *group_padded_offsets,
                                   const int32_t *group_idx_for_bx, int64_t m_blocks,
                                   const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                                   int64_t E, moe_dtype_t dtype, void *h, void *y, int32_t *ready,
                                   int32_t *err_flag, moe_stream_t stream, bool zero_ready) {
    if (!is_half_type(dtype)) return MOE_ERR_UNSUPPORTED;
    if (d_h <= 0 || d_e <= 0 || d_h % 64 != 0 || d_e % 64 != 0) return MOE_ERR_INVALID_ARG;
    if (T <= 0) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0) return MOE_OK;
    moe_status_t st = check_gemm_tables(group_sizes, group_offsets, group_padded_offsets,
                                        group_idx_for_bx, m_blocks, n_rows, E);
    if (st != MOE_OK) return st;
    if (m_blocks > 1088) return MOE_ERR_UNSUPPORTED;
    if (!x || !sorted_token_idx || !q_gate || !q_up || !q_down || !h || !y || !ready)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q_gate) || !aligned16(q_up) || !aligned16(q_down) ||
        !aligned16(h) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (zero_ready) {
        cudaError_t e = cudaMemsetAsync(ready, 0, static_cast<size_t>(m_blocks + 1) * 4, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return cuda_status(moe::launch_grouped_mlp_w4(
        dtype, x, sorted_token_idx, T, q_gate, q_up, q_down, s_gate, s_up, s_down, group_sizes,
        group_offsets, group_padded_offsets, group_idx_for_bx, m_blocks, row_weights, n_rows, d_h, d_e,
        E, h, y, ready, err_flag, s));
}

moe_status_t moe_grouped_mlp_w4a16(const void *x, const int32_t *sorted_token_idx, int64_t T,
                                   const uint8_t *q_gate, const uint8_t *q_up, const uint8_t *q_down,
                                   const float *s_gate, const float *s_up, const float *s_down,
                                   const int32_t *group_sizes, const int32_t *group_offsets,
                                   const int32_t *group_padded_offsets,
                                   const int32_t *group_idx_for_bx, int64_t m_blocks,
                                   const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                                   int64_t E, moe_dtype_t dtype, void *h, void *y, int32_t *ready,
                                   int32_t *err_flag, moe_stream_t stream) {
    return grouped_mlp_w4(x, sorted_token_idx, T, q_gate, q_up, q_down, s_gate, s_up, s_down,
                          group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx, m_blocks,
                          row_weights, n_rows, d_h, d_e, E, dtype, h, y, ready, err_flag, stream, true);
}

// ---------------------------------------------------------------------------
// W4A8: int4 weights x int8 activations, exact int32 sums
// ---------------------------------------------------------------------------
static int64_t w4a8_ws_bytes(int64_t n_rows, int64_t K, int64_t blocks) {
    return static_cast<int64_t>(align_up(static_cast<size_t>(n_rows) * static_cast<size_t>(K) * 2) +
                                align_up(static_cast<size_t>(blocks + 1) * 4));
}

static bool w4a8_k_ok(int64_t K) { return K >= 64 && K % 64 == 0 && K <= (int64_t(1) << 20); }

int64_t moe_gemm_w4a8_workspace_bytes(int64_t M, int64_t K) {
    if (M < 1 || M > 64 || !w4a8_k_ok(K)) return -1;
    return w4a8_ws_bytes(M, K, 1);
}

moe_status_t moe_gemm_w4a8(const int8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K, int32_t *Ct,
                           void *ws, int64_t ws_bytes, int32_t *err_flag, moe_stream_t stream) {
    if (M < 1 || N < 1 || !w4a8_k_ok(K) || N > (int64_t(1) << 24)) return MOE_ERR_INVALID_ARG;
    if (M > 64) return MOE_ERR_UNSUPPORTED;
    if (!A || !B || !Ct || !ws || !aligned16(A) || !aligned16(B) || !aligned16(ws) ||
        (reinterpret_cast<uintptr_t>(Ct) & 3u) != 0)
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_gemm_w4a8_workspace_bytes(M, K)) return MOE_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    void *rows = w;
    int32_t *counters = reinterpret_cast<int32_t *>(w + align_up(static_cast<size_t>(M * K) * 2));
    return cuda_status(moe::launch_gemm_w4a8(A, nullptr, M, B, nullptr, nullptr, nullptr, nullptr, 0, M, M, N,
                                             K, rows, counters, Ct, 1, M, N * M, err_flag,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int64_t moe_grouped_gemm_w4a8_workspace_bytes(int64_t n_rows, int64_t K, int64_t m_blocks) {
    if (n_rows < 1 || m_blocks < 1 || !w4a8_k_ok(K)) return -1;
    return w4a8_ws_bytes(n_rows, K, m_blocks);
}

moe_status_t moe_grouped_gemm_w4a8(const int8_t *x, const int32_t *sorted_token_idx, int64_t T,
                                   const uint8_t *B, const int32_t *group_sizes, const int32_t *group_offsets,
                                   const int32_t *group_padded_offsets, const int32_t *group_idx_for_bx,
                                   int64_t m_blocks, int64_t n_rows, int64_t N, int64_t K, int64_t E,
                                   int32_t *C, void *ws, int64_t ws_bytes, int32_t *err_flag,
                                   moe_stream_t stream) {
    if (T < 1 || N < 1 || !w4a8_k_ok(K) || N > (int64_t(1) << 24)) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0) return MOE_OK;
    if (!sorted_token_idx && n_rows > T) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_gemm_tables(group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                                        m_blocks, n_rows, E);
    if (st != MOE_OK) return st;
    if (m_blocks > 1088) return MOE_ERR_UNSUPPORTED;
    if (!x || !B || !C || !ws || !aligned16(x) || !aligned16(B) || !aligned16(ws) ||
        (reinterpret_cast<uintptr_t>(C) & 3u) != 0)
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_grouped_gemm_w4a8_workspace_bytes(n_rows, K, m_blocks)) return MOE_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    void *rows = w;
    int32_t *counters = reinterpret_cast<int32_t *>(w + align_up(static_cast<size_t>(n_rows * K) * 2));
    return cuda_status(moe::launch_gemm_w4a8(x, sorted_token_idx, T, B, group_sizes, group_offsets,
                                             group_padded_offsets, group_idx_for_bx, m_blocks, 0, n_rows, N, K,
                                             rows, counters, C, N, 1, n_rows * N, err_flag,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

static bool reduce_pair_ok(moe_dtype_t in, moe_dtype_t out, bool allow_fp8) {
    const bool in_ok = in == MOE_F16 || in == MOE_BF16 || in == MOE_F32;
    if (!in_ok) return false;
    if (out == in) return true;
    if (in == MOE_F32 && (out == MOE_F16 || out == MOE_BF16)) return true;
    return allow_fp8 && out == MOE_E4M3;
}

static moe_status_t reduce_common(const void *x, int64_t n_rows, const int32_t *pos,
                                  const float *w, const float *x_sf, const float *sf, int64_t T,
                                  int64_t K, int64_t H, moe_dtype_t in_dtype,
                                  moe_dtype_t out_dtype, void *out, int32_t *err_flag,
                                  moe_stream_t stream, bool allow_fp8, bool pos_early = false) {
    if (T < 0 || K <= 0 || H <= 0 || n_rows < 0) return MOE_ERR_INVALID_ARG;
    if (H % 256 != 0) return MOE_ERR_INVALID_ARG;
    if (!reduce_pair_ok(in_dtype, out_dtype, allow_fp8)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!out || !pos || (n_rows > 0 && !x)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(out) || (x && !aligned16(x))) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_reduce_fused(x, n_rows, pos, w, x_sf, sf, T, K, H, in_dtype,
                                                out_dtype, out, err_flag,
                                                reinterpret_cast<cudaStream_t>(stream), pos_early));
}

moe_status_t moe_reduce_fused(const void *x, int64_t n_rows, const int32_t *token_topk_to_pos,
                              const float *topk_weights, int64_t T, int64_t K, int64_t H,
                              moe_dtype_t in_dtype, moe_dtype_t out_dtype, void *out,
                              int32_t *err_flag, moe_stream_t stream) {
    return reduce_common(x, n_rows, token_topk_to_pos, topk_weights, nullptr, nullptr, T, K, H,
                         in_dtype, out_dtype, out, err_flag, stream, false);
}

moe_status_t moe_reduce_fused_scaled(const void *x, int64_t n_rows,
                                     const int32_t *token_topk_to_pos, const float *topk_weights,
                                     const float *x_sf, const float *sf, int64_t T, int64_t K,
                                     int64_t H, moe_dtype_t in_dtype, moe_dtype_t out_dtype,
                                     void *out, int32_t *err_flag, moe_stream_t stream) {
    return reduce_common(x, n_rows, token_topk_to_pos, topk_weights, x_sf, sf, T, K, H, in_dtype,
                         out_dtype, out, err_flag, stream, true);
}

moe_status_t moe_forward(const void *x, const void *w_g, const float *bias, const void *w_gate,
                         const void *w_up, const void *w_down, int64_t T, int64_t d_h,
                         int64_t d_e, int64_t E, int64_t k, moe_dtype_t dtype, void *ws,
                         size_t ws_bytes, void *out, int32_t *err_flag, moe_stream_t stream) {
    if (!is_half_type(dtype)) return MOE_ERR_UNSUPPORTED;
    if (T < 0 || d_h <= 0 || d_e <= 0 || E <= 0 || k <= 0 || k > E || k > 32 || E > 1024)
        return MOE_ERR_INVALID_ARG;
    if (d_h % 256 != 0 || d_e % 64 != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !w_g || !w_gate || !w_up || !w_down || !out || !ws) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_g)) return MOE_ERR_INVALID_ARG;
    FwdLayout L;
    if (!fwd_layout(T, d_h, d_e, E, k, dtype, &L)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    char *w = static_cast<char *>(ws);
    float *logits = reinterpret_cast<float *>(w + L.off[0]);
    int32_t *topk_idx = reinterpret_cast<int32_t *>(w + L.off[1]);
    float *topk_w = reinterpret_cast<float *>(w + L.off[2]);
    int32_t *sizes = reinterpret_cast<int32_t *>(w + L.off[3]);
    int32_t *offsets = reinterpret_cast<int32_t *>(w + L.off[4]);
    int32_t *padded = reinterpret_cast<int32_t *>(w + L.off[5]);
    int32_t *gidx = reinterpret_cast<int32_t *>(w + L.off[6]);
    int32_t *stok = reinterpret_cast<int32_t *>(w + L.off[7]);
    float *sw = reinterpret_cast<float *>(w + L.off[8]);
    int32_t *pos = reinterpret_cast<int32_t *>(w + L.off[9]);
    void *scratch = w + L.off[10];
    void *A = w + L.off[11];
    void *hbuf = w + L.off[12];
    void *ybuf = w + L.off[13];
    int32_t *ready = reinterpret_cast<int32_t *>(w + L.off[14]);
    const int64_t Tk = T * k;
    const int64_t mb = m_blocks_of(T, k, E, MOE_BLOCK_M);
    moe_status_t st;
    st = gate_topk(x, w_g, bias, T, d_h, E, k, dtype, topk_idx, topk_w, logits,
                   moe_gate_topk_workspace_bytes(T, E), err_flag, stream);
    if (st != MOE_OK) return st;
    // the dispatch also clears the expert MLP's per-block counters
    st = build_dispatch(topk_idx, topk_w, T, k, E, MOE_BLOCK_M, sizes, offsets, padded, gidx, stok,
                        sw, pos, scratch, moe::dispatch_scratch_bytes(Tk, E), ready, stream);
    if (st != MOE_OK) return st;
    if (T <= 64) {
        // every block holds at most 64 rows (a swapped tile of np <= 64 rows):
        // stage 1 gathers them from x, one four-row copy per four of the
        // block's rows (rounded up) per K step.  A
        // full 128-row tile would take 32 such copies per step, which the
        // copy engine issues slower than one tiled copy of the gathered rows
        // (prefill: about 1.9x the expert MLP's time), so larger T first
        // gathers the rows into A.
        st = grouped_mlp(nullptr, w_gate, w_up, w_down, sizes, offsets, padded, gidx, mb, nullptr, Tk,
                         d_h, d_e, E, dtype, hbuf, ybuf, ready, err_flag, stream, false, x, stok, T);
    } else {
        // the rows of A in token order: each token's row read once, written to
        // its k rows (the row-order gather re-read token rows from DRAM about
        // seven times at prefill: 409 MB for 58.7 MB of tokens)
        st = moe_gather_rows_by_token(x, pos, T, k, Tk, d_h, dtype, A, err_flag, stream);
        if (st != MOE_OK) return st;
        st = grouped_mlp(A, w_gate, w_up, w_down, sizes, offsets, padded, gidx, mb, nullptr, Tk, d_h,
                         d_e, E, dtype, hbuf, ybuf, ready, err_flag, stream, false);
    }
    if (st != MOE_OK) return st;
    // the combine's positions and weights come from the dispatch, which
    // completed before the expert MLP passed its own dependency wait
    return reduce_common(ybuf, Tk, pos, topk_w, nullptr, nullptr, T, k, d_h, dtype, dtype, out, err_flag,
                         stream, false, true);
}

moe_status_t moe_forward_w4a16(const void *x, const void *w_g, const float *bias,
                               const uint8_t *q_gate, const uint8_t *q_up, const uint8_t *q_down,
                               const float *s_gate, const float *s_up, const float *s_down,
                               int64_t T, int64_t d_h, int64_t d_e, int64_t E, int64_t k,
                               moe_dtype_t dtype, void *ws, size_t ws_bytes, void *out,
                               int32_t *err_flag, moe_stream_t stream) {
    if (!is_half_type(dtype)) return MOE_ERR_UNSUPPORTED;
    if (T < 0 || d_h <= 0 || d_e <= 0 || E <= 0 || k <= 0 || k > E || k > 32 || E > 1024)
        return MOE_ERR_INVALID_ARG;
    if (d_h % 256 != 0 || d_e % 64 != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (m_blocks_of(T, k, E, MOE_BLOCK_M) > 1088) return MOE_ERR_UNSUPPORTED;
    if (!x || !w_g || !q_gate || !q_up || !q_down || !out || !ws) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_g)) return MOE_ERR_INVALID_ARG;
    FwdLayout L;
    if (!fwd_layout(T, d_h, d_e, E, k, dtype, &L)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    char *w = static_cast<char *>(ws);
    float *logits = reinterpret_cast<float *>(w + L.off[0]);
    int32_t *topk_idx = reinterpret_cast<int32_t *>(w + L.off[1]);
    float *topk_w = reinterpret_cast<float *>(w + L.off[2]);
    int32_t *sizes = reinterpret_cast<int32_t *>(w + L.off[3]);
    int32_t *offsets = reinterpret_cast<int32_t *>(w + L.off[4]);
    int32_t *padded = reinterpret_cast<int32_t *>(w + L.off[5]);
    int32_t *gidx = reinterpret_cast<int32_t *>(w + L.off[6]);
    int32_t *stok = reinterpret_cast<int32_t *>(w + L.off[7]);
    float *sw = reinterpret_cast<float *>(w + L.off[8]);
    int32_t *pos = reinterpret_cast<int32_t *>(w + L.off[9]);
    void *scratch = w + L.off[10];
    void *hbuf = w + L.off[12];
    void *ybuf = w + L.off[13];
    int32_t *ready = reinterpret_cast<int32_t *>(w + L.off[14]);
    const int64_t Tk = T * k;
    const int64_t mb = m_blocks_of(T, k, E, MOE_BLOCK_M);
    moe_status_t st = gate_topk(x, w_g, bias, T, d_h, E, k, dtype, topk_idx, topk_w, logits,
                                moe_gate_topk_workspace_bytes(T, E), err_flag, stream);
    if (st != MOE_OK) return st;
    st = build_dispatch(topk_idx, topk_w, T, k, E, MOE_BLOCK_M, sizes, offsets, padded, gidx, stok,
                        sw, pos, scratch, moe::dispatch_scratch_bytes(Tk, E), ready, stream);
    if (st != MOE_OK) return st;
    st = grouped_mlp_w4(x, stok, T, q_gate, q_up, q_down, s_gate, s_up, s_down, sizes, offsets,
                        padded, gidx, mb, nullptr, Tk, d_h, d_e, E, dtype, hbuf, ybuf, ready, err_flag,
                        stream, false);
    if (st != MOE_OK) return st;
    // the combine's positions and weights come from the dispatch, which
    // completed before the expert MLP passed its own dependency wait
    return reduce_common(ybuf, Tk, pos, topk_w, nullptr, nullptr, T, k, d_h, dtype, dtype, out, err_flag,
                         stream, false, true);
}


}  // extern "C"

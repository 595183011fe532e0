// grouped_gemm_w4.cu -- the expert MLP (both GEMM stages in one launch) with
// int4 weights and 16-bit activations (weight-only W4A16), built for decode
// (blocks of up to 64 rows, where the expert weights are read once per step
// and their bytes are the whole cost; larger blocks are split into 64-row
// units), and the W4A8 GEMM on the same machinery.
//
// Weight format (TileLang tutorial ch.18 skeletons.py, w4a8_dequant_gemm):
// int4 values two per byte, element j of a row in byte j/2 at nibble j%2
// from the low end, two's complement; the kernel unpacks them on chip and
// casts them to the compute type before the GEMM (the module notes: the same
// kernel with 16-bit activations is the weight-only W4A16 form).  Reading: an
// optional fp32 scale per output channel multiplies the fp32 sum.
//
// launch_pack_int4 rewrites a stacked [E, N, K] weight in that format into
// tiles of R output channels (R = 128 for W_gate / W_up, 256 for W_down):
// [E][ceil(N/R)][K/64][R rows][32 bytes], so that the 64-wide K step of one
// tile is one contiguous block (one bulk copy, sequential DRAM reads), rows
// past N holding zeros.  Inside each 32-bit word (8 elements) elements 2m
// and 2m+1 move to nibbles m and m+4, stored offset-binary (value + 8), so
// one AND-OR with the fp16 (or bf16) exponent of 1024 (128) and one packed
// subtraction of 1032 (136) give two exact values.
//
// Kernel (one persistent CTA per SM, 480 threads):
//   warp 0      producer: per 128-wide K step (two 64-wide sub-steps), one
//               stage of a 6-deep ring: the block's rows (stage 1: up to 64
//               token rows gathered from x by four-row TMA gathers; stage 2:
//               64 rows of h) and the packed weights of 256 output channels
//               (16 KB, bulk copies of contiguous tile blocks);
//   warps 6..13 converters: unpack the stage's 256 x 64 weights straight into
//               tensor memory (tcgen05.st; thread = TMEM lane = output
//               channel), one of two 128-column A buffers;
//   warps 1, 14 MMA: tcgen05.mma M=128 N=rows with the A operand (the
//               weights, one 128-channel half per warp, the two halves issued
//               in parallel) read from tensor memory and the block's rows as
//               the shared-memory B operand, into a TMEM accumulator, double
//               buffered.  Unpacking into tensor memory
//               keeps the 16-bit weights off shared memory: per step only the
//               8 KB of packed weights and the rows pass through it;
//   warps 2..5  epilogue: scales, silu(gate)*up for stage 1, row-masked
//               stores; a stage-1 warp-tile publishes its h rows on the
//               block's counter for the stage-2 tiles.
// Tiles are taken as in the 16-bit expert MLP: every tile, the first
// included, from a shared counter, stage-1 tiles before stage-2 tiles, over
// units of at most 64 rows (a dispatch block with more rows is two units);
// a stage-2 tile waits (bounded) until its block's counter shows every
// stage-1 warp-tile of the block stored.  Every wait is bounded; on a
// timeout the kernel records MOE_ERR_TIMEOUT, lets its copies and MMAs land,
// frees TMEM and returns.
//
// W4A8 (int4 weights x int8 activations, exact int32 sums):
//   * the GEMM form of the same kernel: stage-2 tiles only (256 channels x
//     one K chunk of at most 16384), rows from an fp16 copy of the int8
//     activations (w4a8_rows_kernel), an int32 epilogue; every fp32 partial
//     sum is an integer of magnitude <= 2^24, so it is exact, and the chunks
//     are added with integer atomics;
//   * w4a8_gemv_kernel for the dense form with at most 8 rows: the weights
//     streamed through a shared-memory ring into the CUDA cores, dp4a on the
//     packed bytes.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int W4_BK = 64;                        // K elements per sub-step (one packed block)
constexpr int W4_SUB = 2;                        // sub-steps per pipeline stage (K = 128)
constexpr int W4_ROWS = 256;                     // weight rows (output channels) per tile
constexpr int W4_PACK_ROW = W4_BK / 2;           // 32 packed bytes per row and sub-step
constexpr int W4_PACK_SUB = W4_ROWS * W4_PACK_ROW;      // 8 KB
constexpr int W4_PACK_BYTES = W4_SUB * W4_PACK_SUB;     // 16 KB
constexpr int W4_TOK_ROWS = 64;                  // the most rows a block may hold here
constexpr int W4_TOK_SUB = W4_TOK_ROWS * W4_BK * 2;     // 8 KB, 128-byte swizzled
constexpr int W4_TOK_BYTES = W4_SUB * W4_TOK_SUB;       // 16 KB
constexpr int W4_STAGE_BYTES = W4_TOK_BYTES + W4_PACK_BYTES;
constexpr int W4_STAGES = 6;
constexpr int W4_CONVS = 2;                      // A buffers in tensor memory
constexpr int W4_A_SUB = W4_BK;                  // columns per sub-step: 2 halves x 64 x 16-bit / 32-bit
constexpr int W4_A_COLS = W4_SUB * W4_A_SUB;
constexpr int W4_A_COL0 = 256;                   // A buffers after the two accumulators
constexpr int W4_THREADS = 480;
constexpr int W4_CONV_WARP0 = 6;                 // converter warps 6..13: two per TMEM lane quarter
constexpr int W4_CONV_WARPS = 8;
constexpr int W4_EPI_WARPS = 4;
constexpr int W4_MMA2_WARP = 14;                 // issues the second 128-channel half's MMAs
constexpr int W4_MMA_WARPS = 2;
constexpr int W4_TRING = 4;
constexpr int W4_NEXT_FETCH = 1;                 // stages before a tile's end that the next one is taken
constexpr int W4_ACC_COLS = 128;                 // 2 x up to 64 columns per accumulator
constexpr int W4_TMEM_COLS = 512;
static_assert(W4_A_COL0 + W4_CONVS * W4_A_COLS <= W4_TMEM_COLS && 2 * W4_ACC_COLS <= W4_A_COL0, "tmem");
static_assert(W4_STAGES > W4_CONVS, "a stage is released W4_CONVS steps after its use");
constexpr int W4_MAX_BLOCKS = 1088;              // M blocks the schedule lists
constexpr int W4_BAR_BYTES = 512;
// the unit list (up to two 64-row units per block), then per block its
// expert, first row and row count, then the scan's scratch
constexpr int W4_SCHED_BYTES = W4_MAX_BLOCKS * (2 * 4 + 4 * 2 + 1) + 64 * 4;
constexpr int W4_XPOSE_BYTES = W4_EPI_WARPS * 32 * 17 * 4;  // W4A8 epilogue: a 32 x 16 transpose per warp
constexpr int W4_SMEM_BYTES = 1024 + W4_STAGES * W4_STAGE_BYTES + W4_BAR_BYTES + W4_SCHED_BYTES + W4_XPOSE_BYTES;
static_assert(W4_SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(W4_STAGE_BYTES % 1024 == 0, "swizzle atoms");

// ---------------------------------------------------------------------------
// repack: one thread per 32-bit output word (8 elements)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t w4_reorder(uint32_t w) {
    uint32_t o = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t nib = (w >> (4 * e)) & 0xFu;
        const int slot = (e & 1) ? 4 + (e >> 1) : (e >> 1);
        o |= nib << (4 * slot);
    }
    return o ^ 0x88888888u;  // offset-binary: value + 8
}

// plain [E, N, K/2] bytes -> [E][NT = ceil(N/R)][S = K/64][R][32 bytes]
__global__ void pack_int4_kernel(const uint32_t *__restrict__ plain, int64_t E, int64_t N, int64_t K,
                                 int R, uint32_t *__restrict__ packed) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t NT = (N + R - 1) / R, S = K / W4_BK;
    const int64_t total = E * NT * S * R * 8;  // output words
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int w = static_cast<int>(i & 7);
    int64_t rest = i >> 3;
    const int r = static_cast<int>(rest % R);
    rest /= R;
    const int64_t st = rest % S;
    rest /= S;
    const int64_t t = rest % NT;
    const int64_t e = rest / NT;
    const int64_t n = t * R + r;
    packed[i] = n < N ? w4_reorder(plain[(e * N + n) * (K / 8) + st * 8 + w]) : 0x88888888u;  // zeros past N
}

struct W4Params {
    const int32_t *sizes, *offsets, *padded, *gidx;
    const int32_t *gather_idx;  // stage-1 rows: token indices into x
    const uint8_t *q_gate, *q_up, *q_down;  // tiled packed weights (see launch_pack_int4)
    const float *row_weights;
    const float *s_gate, *s_up, *s_down;
    int *ready;         // per M block: stage-1 epilogue warp-tiles stored
    int *tile_counter;  // next tile beyond the first wave
    void *h, *y;
    int m_blocks, d_h, d_e;
    int nt0, nt1;       // output tiles per block: stage 1 (128 columns), stage 2 (256)
    int kb0, kb1;       // 64-wide K sub-steps: stage 1 (d_h / 64), stage 2 (d_e / 64)
    int *err;
    // W4A8 GEMM form (nt0 = 0: stage-2 tiles only, rows from h, int32 out):
    // a stage-2 tile covers sub-steps [kc * kchunk, (kc + 1) * kchunk) of
    // kb1; ksplit = 1 and kchunk = kb1 for the expert MLP
    int ksplit, kchunk;
    int dense_rows;        // > 0: one block of this many rows, no tables
    int32_t *out_i32;      // non-null: int32 results at m * ld_row + n * ld_col
    int64_t ld_row, ld_col;
    int atomic_out;        // add (the K chunks of a tile) instead of store
};

struct W4Tile {
    int g, m_start, rows, n0, bx, phase, kc;
};

// Tile t of the launch: the stage-1 tiles of every listed unit first, then
// the stage-2 tiles in the same unit order.  A unit is up to 64 rows: a
// 128-row block of the tables with more than 64 rows is two units (list
// entry 2 bx + half), so the kernel serves any number of tokens.
__device__ __forceinline__ W4Tile w4_tile(const W4Params &p, const int *list, const int *blk_g,
                                          const int *blk_m, const uint8_t *blk_rows, int n_units,
                                          int t) {
    W4Tile ti;
    const int n0_tiles = n_units * p.nt0;
    int pos, nt;
    if (t < n0_tiles) {
        ti.phase = 0;
        ti.kc = 0;
        pos = t / p.nt0;
        nt = t - pos * p.nt0;
        ti.n0 = nt * 128;
    } else {
        ti.phase = 1;
        t -= n0_tiles;
        const int per_block = p.nt1 * p.ksplit;
        pos = t / per_block;
        const int rem = t - pos * per_block;
        nt = rem / p.ksplit;
        ti.kc = rem - nt * p.ksplit;
        ti.n0 = nt * 256;
    }
    const int e = list[pos];
    const int bx = e >> 1, half = e & 1;
    ti.bx = bx;
    ti.g = blk_g[bx];
    ti.m_start = blk_m[bx] + half * W4_TOK_ROWS;
    ti.rows = min(static_cast<int>(blk_rows[bx]) - half * W4_TOK_ROWS, W4_TOK_ROWS);
    return ti;
}

// stage-1 epilogue warp-tiles that publish on block bx's counter: every
// unit of the block, so a stage-2 tile of either unit waits for both
__device__ __forceinline__ int w4_ready_target(const W4Params &p, const uint8_t *blk_rows, int bx) {
    return W4_EPI_WARPS * p.nt0 * (blk_rows[bx] > W4_TOK_ROWS ? 2 : 1);
}

// 64-wide K sub-steps of a tile (its K chunk for a stage-2 tile)
__device__ __forceinline__ int w4_ksub(const W4Params &p, const W4Tile &ti) {
    if (ti.phase == 0) return p.kb0;
    const int left = p.kb1 - ti.kc * p.kchunk;
    return left < p.kchunk ? left : p.kchunk;
}

// bulk copy of `bytes` contiguous bytes (16-byte aligned) into shared memory,
// completing on `bar`, with an L2 policy
__device__ __forceinline__ void w4_bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                            uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void w4_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long start = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - start > kWaitTimeoutNs) return;
}

// Unpack one 32-bit word (8 elements, the repacked layout) into 8 values of
// the compute type, in element order.  fp16: nibbles at bits 0 and 16 OR-ed
// into the mantissa of 1024 give 1024 + u (then minus 1032); nibbles at bits
// 4 and 20 give 1024 + 16 u (then times 1/16 minus 72), so only the pairs
// of the upper byte need a shift.  bf16 has 7 mantissa bits: every pair is
// shifted down to bit 0 and 136 subtracted from 128 + u.
template <int DT>
__device__ __forceinline__ uint4 w4_unpack8(uint32_t w) {
    constexpr uint32_t MAGIC = DT == kBF16 ? 0x43004300u : 0x64006400u;  // 128 / 1024, twice
    uint4 r;
    if constexpr (DT == kF16) {
        const uint32_t w8 = w >> 8;
        uint32_t q[4];
        q[0] = (w & 0x000F000Fu) | MAGIC;
        q[1] = (w & 0x00F000F0u) | MAGIC;
        q[2] = (w8 & 0x000F000Fu) | MAGIC;
        q[3] = (w8 & 0x00F000F0u) | MAGIC;
        const __half2 off = __floats2half2_rn(1032.0f, 1032.0f);
        const __half2 sixteenth = __floats2half2_rn(0.0625f, 0.0625f), off16 = __floats2half2_rn(-72.0f, -72.0f);
        const __half2 v0 = __hsub2(*reinterpret_cast<__half2 *>(&q[0]), off);
        const __half2 v1 = __hfma2(*reinterpret_cast<__half2 *>(&q[1]), sixteenth, off16);
        const __half2 v2 = __hsub2(*reinterpret_cast<__half2 *>(&q[2]), off);
        const __half2 v3 = __hfma2(*reinterpret_cast<__half2 *>(&q[3]), sixteenth, off16);
        r = make_uint4(*reinterpret_cast<const uint32_t *>(&v0), *reinterpret_cast<const uint32_t *>(&v1),
                       *reinterpret_cast<const uint32_t *>(&v2), *reinterpret_cast<const uint32_t *>(&v3));
    } else {
        uint32_t q[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) q[m] = ((w >> (4 * m)) & 0x000F000Fu) | MAGIC;
        const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
        __nv_bfloat162 v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&q[m]), off);
        r = make_uint4(*reinterpret_cast<uint32_t *>(&v[0]), *reinterpret_cast<uint32_t *>(&v[1]),
                       *reinterpret_cast<uint32_t *>(&v[2]), *reinterpret_cast<uint32_t *>(&v[3]));
    }
    return r;
}

// 32 lanes x 32 bit, 64 consecutive columns from thread i's 64 registers into lane (base + i).
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, "
        "%33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, "
        "%49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]),
        "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]),
        "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]),
        "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]),
        "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}
// One channel's 64 packed weights of a sub-step (32 bytes of shared memory)
// unpacked into 32 words of two 16-bit values, in element order.
template <int DT>
__device__ __forceinline__ void w4_unpack_row(const uint8_t *prow, uint32_t *cols) {
    const uint4 lo = *reinterpret_cast<const uint4 *>(prow);
    const uint4 hi = *reinterpret_cast<const uint4 *>(prow + 16);
    const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint4 v = w4_unpack8<DT>(wv[w]);
        cols[4 * w + 0] = v.x;
        cols[4 * w + 1] = v.y;
        cols[4 * w + 2] = v.z;
        cols[4 * w + 3] = v.w;
    }
}

// Exclusive scan of one int per thread across the CTA; returns the total.
__device__ __forceinline__ int w4_cta_scan(int v, int *scratch, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < W4_THREADS / 32; ++w) {
        const int x = scratch[w];
        if (w < warp) base += x;
        tot += x;
    }
    __syncthreads();
    *total = tot;
    return base + incl - v;
}

template <int DT>
__global__ void __launch_bounds__(W4_THREADS, 1)
    grouped_mlp_w4_kernel(const __grid_constant__ CUtensorMap tmX,    // x [T, d_h], box 64 x 1
                          const __grid_constant__ CUtensorMap tmH,    // h [rows, d_e], box 64 x 64
                          const W4Params p) {
    using OutT = typename Elem<DT>::T;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *stages = smem;                                     // [W4_STAGES][tokens 8 KB | packed 8 KB]
    uint64_t *bars = reinterpret_cast<uint64_t *>(stages + W4_STAGES * W4_STAGE_BYTES);
    // barriers: pfull, pempty [stages]; cfull, cempty [convs]; tfull, tempty [2]; tidf, tide [ring]
    constexpr int NBARS = 2 * W4_STAGES + 2 * W4_CONVS + 4 + 2 * W4_TRING;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *tid_ring = reinterpret_cast<int *>(tmem_slot + 2);
    // per stage: 16 * gemm stage + sub-steps held (1 or 2); 0 = no more stages
    volatile int *stage_flag = reinterpret_cast<volatile int *>(tid_ring + W4_TRING);
    static_assert(NBARS * 8 + 8 + 4 * W4_TRING + 4 * W4_STAGES <= W4_BAR_BYTES, "barrier area");
    int *list = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + W4_BAR_BYTES);
    int *blk_g = list + 2 * W4_MAX_BLOCKS;
    int *blk_m = blk_g + W4_MAX_BLOCKS;
    uint8_t *blk_rows = reinterpret_cast<uint8_t *>(blk_m + W4_MAX_BLOCKS);
    int *scan_scratch = reinterpret_cast<int *>(blk_rows + W4_MAX_BLOCKS);
    int *xpose = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + W4_BAR_BYTES + W4_SCHED_BYTES);
    static_assert(W4_MAX_BLOCKS % 4 == 0, "scratch alignment");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = smem_u32(bars);
    auto pfull = [&](int s) { return bar0 + 8u * s; };
    auto pempty = [&](int s) { return bar0 + 8u * (W4_STAGES + s); };
    auto cfull = [&](int c) { return bar0 + 8u * (2 * W4_STAGES + c); };
    auto cempty = [&](int c) { return bar0 + 8u * (2 * W4_STAGES + W4_CONVS + c); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * W4_STAGES + 2 * W4_CONVS + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * W4_STAGES + 2 * W4_CONVS + 2 + a); };
    auto tidf = [&](int i) { return bar0 + 8u * (2 * W4_STAGES + 2 * W4_CONVS + 4 + i); };
    auto tide = [&](int i) { return bar0 + 8u * (2 * W4_STAGES + 2 * W4_CONVS + 4 + W4_TRING + i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < W4_STAGES; ++s) {
            mbar_init(pfull(s), 1);
            // every converter warp, once both it and the MMA are done with the
            // stage (see the converters: one MMA commit per step, not two)
            mbar_init(pempty(s), W4_CONV_WARPS);
        }
        for (int c = 0; c < W4_CONVS; ++c) {
            mbar_init(cfull(c), W4_CONV_WARPS);
            mbar_init(cempty(c), W4_MMA_WARPS);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull(a), W4_MMA_WARPS);
            mbar_init(tempty(a), W4_EPI_WARPS);
        }
        for (int i = 0; i < W4_TRING; ++i) {
            mbar_init(tidf(i), 1);
            mbar_init(tide(i), W4_MMA_WARPS + W4_EPI_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmH);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), W4_TMEM_COLS);
        tmem_relinquish();
    }
    griddep_wait();  // the tables, x and the counters come from earlier kernels
    griddep_launch_dependents();
    // every tile, the first included, comes from the shared counter (see the
    // producer); the first claim's round trip hides behind the schedule build
    int first_tile = 0;
    if (threadIdx.x == 0) first_tile = atomicAdd(p.tile_counter, 1);

    // ----- schedule: the units of the non-empty M blocks in order -----
    int n_blocks = 0;  // units
    if (p.dense_rows > 0) {  // one block: rows 0 .. dense_rows - 1, weight 0
        n_blocks = 1;
        if (threadIdx.x == 0) {
            list[0] = 0;
            blk_g[0] = 0;
            blk_m[0] = 0;
            blk_rows[0] = static_cast<uint8_t>(p.dense_rows);
        }
    } else {
        const int chunk = (p.m_blocks + W4_THREADS - 1) / W4_THREADS;
        const int lo = threadIdx.x * chunk, hi = min(p.m_blocks, lo + chunk);
        int mine = 0;
        for (int bx = lo; bx < hi; ++bx) {
            const int g = __ldg(p.gidx + bx);
            const int rel = bx * 128 - __ldg(p.padded + g);
            int rows = __ldg(p.sizes + g) - rel;
            rows = rows < 0 ? 0 : (rows > 128 ? 128 : rows);
            blk_g[bx] = g;
            blk_m[bx] = rel + __ldg(p.offsets + g);
            blk_rows[bx] = static_cast<uint8_t>(rows);
            mine += (rows > 0) + (rows > W4_TOK_ROWS);
        }
        int base = w4_cta_scan(mine, scan_scratch, &n_blocks);
        for (int bx = lo; bx < hi; ++bx) {
            if (blk_rows[bx] > 0) list[base++] = 2 * bx;
            if (blk_rows[bx] > W4_TOK_ROWS) list[base++] = 2 * bx + 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = n_blocks * (p.nt0 + p.nt1 * p.ksplit);

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        // the whole warp: lane 0 takes tiles, arms the stage barriers and
        // issues the weight copies; lane j (< rows / 4) holds the token ids
        // of rows 4j .. 4j+3 for the tile and issues their gather every step
        const uint64_t pol_first = l2_policy_evict_first();  // weights are read once
        int stage = 0;
        uint32_t phase = 0;
        long issued = 0;
        bool ok = true;
        int rslot = 0;
        uint32_t rphase = 0;
        // the next tile is taken W4_NEXT_FETCH stages before the current tile's
        // last copy (at the end of the launch the last tiles then go to CTAs
        // that are about to be free; the atomic's result is first used at the
        // next tile, so its round trip stays hidden)
        // Tiles are taken in order and stage-1 tiles precede stage-2 tiles, so a
        // stage-2 tile's stage-1 tiles are all held by running CTAs when it is
        // taken: progress does not need the whole grid resident at once.
        int next_tile = first_tile;
        bool have_next = true;
        for (int it = 0; ok; ++it) {
            int tile = 0;
            int go = 1;
            if (lane == 0) {
                if (!have_next) next_tile = atomicAdd(p.tile_counter, 1);
                tile = next_tile;
                have_next = false;
                if (tile >= total) tile = -1;
                go = mbar_wait_bounded(tide(rslot), rphase ^ 1u, abort_flag, p.err) ? 1 : 0;
                if (go) {
                    tid_ring[rslot] = tile;
                    mbar_arrive(tidf(rslot));
                }
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (++rslot == W4_TRING) {
                rslot = 0;
                rphase ^= 1u;
            }
            if (!go) {
                ok = false;
                break;
            }
            if (tile < 0) break;
            const W4Tile ti = w4_tile(p, list, blk_g, blk_m, blk_rows, n_blocks, tile);
            // stage 2 reads its block's h rows: all stage-1 warp-tiles stored
            if (ti.phase == 1 && p.nt0 > 0) {
                if (lane == 0)
                    go = counter_wait_bounded(p.ready + ti.bx, w4_ready_target(p, blk_rows, ti.bx), abort_flag,
                                              p.err) ? 1 : 0;
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
            }
            int np = (ti.rows + 15) & ~15;
            if (np > W4_TOK_ROWS) {  // units hold at most 64 rows
                np = W4_TOK_ROWS;
                if (lane == 0 && p.err) atomicExch(p.err, kErrDeviceFlag);
            }
            // this lane's four token ids (rows past the block repeat its first row)
            int i0 = 0, i1 = 0, i2 = 0, i3 = 0;
            const bool gatherer = ti.phase == 0 && 4 * lane < np;
            if (gatherer) {
                const int32_t *ids = p.gather_idx + ti.m_start;
                const int r = 4 * lane;
                i0 = __ldg(ids + (r < ti.rows ? r : 0));
                i1 = __ldg(ids + (r + 1 < ti.rows ? r + 1 : 0));
                i2 = __ldg(ids + (r + 2 < ti.rows ? r + 2 : 0));
                i3 = __ldg(ids + (r + 3 < ti.rows ? r + 3 : 0));
            }
            const int ksub = w4_ksub(p, ti);
            const int kbase = ti.kc * p.kchunk;  // first sub-step of the tile's K chunk
            const int kstages = (ksub + W4_SUB - 1) / W4_SUB;
            const int fetch_kb = kstages > W4_NEXT_FETCH ? kstages - W4_NEXT_FETCH : 0;
            for (int kb = 0; kb < kstages; ++kb) {
                if (lane == 0 && kb == fetch_kb) {
                    next_tile = atomicAdd(p.tile_counter, 1);
                    have_next = true;
                }
                const int nsub = min(W4_SUB, ksub - kb * W4_SUB);
                const uint32_t tx = static_cast<uint32_t>(nsub * ((ti.phase == 0 ? np * W4_BK * 2 : W4_TOK_SUB) +
                                                                  W4_PACK_SUB));
                if (lane == 0) go = mbar_wait_bounded(pempty(stage), phase ^ 1u, abort_flag, p.err) ? 1 : 0;
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
                uint8_t *st = stages + stage * W4_STAGE_BYTES;
                const uint32_t tok = smem_u32(st), pk = smem_u32(st + W4_TOK_BYTES);
                const uint32_t fb = pfull(stage);
                if (lane == 0) {
                    stage_flag[stage] = 16 * ti.phase + nsub;
                    mbar_arrive_expect_tx(fb, tx);
                }
                __syncwarp();  // the stage's byte count is armed before any copy lands
                const int sub0 = kbase + kb * W4_SUB;  // first 64-wide sub-step of the stage
                if (ti.phase == 0) {
                    if (gatherer)
                        for (int u = 0; u < nsub; ++u)
                            tma_gather4(tok + static_cast<uint32_t>(u * W4_TOK_SUB + 4 * lane * W4_BK * 2), &tmX, fb,
                                        (sub0 + u) * W4_BK, i0, i1, i2, i3);
                    if (lane == 0) {
                        // 128 gate rows for each sub-step, then 128 up rows (consecutive blocks)
                        const int64_t blk = (static_cast<int64_t>(ti.g) * p.nt0 + ti.n0 / 128) * p.kb0 + sub0;
                        const uint32_t bytes = static_cast<uint32_t>(nsub * W4_PACK_SUB / 2);
                        w4_bulk_g2s(pk, p.q_gate + blk * (W4_PACK_SUB / 2), bytes, fb, pol_first);
                        w4_bulk_g2s(pk + W4_PACK_BYTES / 2, p.q_up + blk * (W4_PACK_SUB / 2), bytes, fb, pol_first);
                    }
                } else if (lane == 0) {
                    for (int u = 0; u < nsub; ++u)
                        tma_load_2d(tok + static_cast<uint32_t>(u * W4_TOK_SUB), &tmH, fb, (sub0 + u) * W4_BK,
                                    ti.m_start);
                    const int64_t blk = (static_cast<int64_t>(ti.g) * p.nt1 + ti.n0 / 256) * p.kb1 + sub0;
                    w4_bulk_g2s(pk, p.q_down + blk * W4_PACK_SUB, static_cast<uint32_t>(nsub * W4_PACK_SUB), fb,
                                pol_first);
                }
                ++issued;
                if (++stage == W4_STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0) {
            if (ok && mbar_wait_bounded(pempty(stage), phase ^ 1u, abort_flag, p.err)) {
                stage_flag[stage] = 0;  // the converters stop here
                mbar_arrive(pfull(stage));
            }
            if (!ok) {
                // let every copy still in flight land before shared memory goes away
                for (long j = 1; j <= W4_STAGES && j <= issued; ++j) {
                    const long i = issued - j;
                    w4_wait_drain(pfull(static_cast<int>(i % W4_STAGES)),
                                  static_cast<uint32_t>((i / W4_STAGES) & 1));
                }
            }
        }
    } else if (warp == 1 || warp == W4_MMA2_WARP) {
        // --------------------------------- MMA ---------------------------------
        // warp 1 issues the MMAs of channels 0..127, warp 14 those of 128..255:
        // two independent accumulator chains, issued in parallel (one thread
        // issues an MMA about every 85 cycles, whatever its size)
        const int half = warp == 1 ? 0 : 1;
        if (lane == 0) {
            int stage = 0, cb = 0;
            uint32_t phase = 0, cph = 0;
            int local = 0;
            bool ok = true;
            uint32_t last_bar = 0, last_parity = 0;
            bool committed = false;
            int rslot = 0;
            uint32_t rphase = 0;
            for (;;) {
                if (!mbar_wait_bounded(tidf(rslot), rphase, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const int tile = tid_ring[rslot];
                mbar_arrive(tide(rslot));
                if (++rslot == W4_TRING) {
                    rslot = 0;
                    rphase ^= 1u;
                }
                if (tile < 0) break;
                const W4Tile ti = w4_tile(p, list, blk_g, blk_m, blk_rows, n_blocks, tile);
                const int ksub = w4_ksub(p, ti);
                const int kstages = (ksub + W4_SUB - 1) / W4_SUB;
                const int acc = local & 1;
                const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
                if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                int np = (ti.rows + 15) & ~15;
                if (np > W4_TOK_ROWS) np = W4_TOK_ROWS;
                // D[channel][row]: channels 0..127 into columns [0, np), 128..255 into [np, 2np)
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * W4_ACC_COLS + half * np);
                const uint32_t idesc = idesc_f16(DT == kBF16, 128, static_cast<uint32_t>(np));
                for (int kb = 0; kb < kstages; ++kb) {
                    const int nsub = min(W4_SUB, ksub - kb * W4_SUB);
                    if (!mbar_wait_bounded(cfull(cb), cph, abort_flag, p.err) ||
                        !mbar_wait_bounded(pfull(stage), phase, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int u = 0; u < nsub; ++u) {
                        // A buffer cb: channels 0..127 in columns [0, 64) (sub-step u at 32 u),
                        // 128..255 in [64, 128)
                        const uint32_t a0 = tmem_base + static_cast<uint32_t>(W4_A_COL0 + cb * W4_A_COLS +
                                                                              half * W4_A_SUB + u * (W4_A_SUB / 2));
                        const uint64_t bd = smem_desc_sw128(smem_u32(stages + stage * W4_STAGE_BYTES + u * W4_TOK_SUB));
#pragma unroll
                        for (int k = 0; k < W4_BK / 16; ++k) {
                            const uint32_t accum = (kb | u | k) != 0 ? 1u : 0u;
                            tc_mma_f16_ta(d_tmem, a0 + 8u * k, bd + 2u * k, idesc, accum);
                        }
                    }
                    // the unpacked weights may be overwritten once these finish; the
                    // converters then also release this step's stage for the producer
                    tc_commit(cempty(cb));
                    last_bar = cempty(cb);
                    last_parity = cph;
                    committed = true;
                    if (++stage == W4_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++cb == W4_CONVS) {
                        cb = 0;
                        cph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(tfull(acc));
                ++local;
            }
            if (!ok && committed) w4_wait_drain(last_bar, last_parity);
        }
    } else if (warp >= W4_CONV_WARP0 && warp < W4_CONV_WARP0 + W4_CONV_WARPS) {
        // ------------------------------ converters ------------------------------
        // warp w owns TMEM lanes 32 (w % 4) .. +31: its thread t unpacks the
        // 64 weights of channel 32 (w % 4) + t of half (w - 6) / 4 (channels
        // 0..127 in columns [0, 32) of the A buffer, 128..255 in [32, 64))
        const int quarter = warp & 3;
        const int half = (warp - W4_CONV_WARP0) / 4;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        int stage = 0, cb = 0;
        uint32_t phase = 0, cph = 0;
        long step = 0;
        for (;;) {
            if (!mbar_wait_bounded(pfull(stage), phase, abort_flag, p.err)) break;
            const int flag = stage_flag[stage];
            if (flag == 0) break;
            const int nsub = flag & 15, gphase = flag >> 4;
            if (!mbar_wait_bounded(cempty(cb), cph ^ 1u, abort_flag, p.err)) break;
            // the buffer is free: the MMA has finished step - W4_CONVS, whose
            // stage (rows and packed weights, both read) goes back to the producer
            if (step >= W4_CONVS && lane == 0)
                mbar_arrive(pempty((stage + W4_STAGES - W4_CONVS) % W4_STAGES));
            tc_fence_after();
            // packed rows: stage 1 [gate sub 0 | gate sub 1 | up sub 0 | up sub 1] (4 KB
            // each), stage 2 [sub 0 | sub 1] (8 KB each, channels 0..255)
            const uint8_t *pk = stages + stage * W4_STAGE_BYTES + W4_TOK_BYTES;
            const int ch = quarter * 32 + lane;  // channel within the half
            const uint8_t *prow = gphase == 0 ? pk + half * (W4_PACK_BYTES / 2) + ch * W4_PACK_ROW
                                              : pk + (half * 128 + ch) * W4_PACK_ROW;
            const int sub_stride = gphase == 0 ? W4_PACK_SUB / 2 : W4_PACK_SUB;
            // the half's columns of both sub-steps are adjacent: one store of 64 columns
            const uint32_t a_dst =
                tmem_base + lane_base + static_cast<uint32_t>(W4_A_COL0 + cb * W4_A_COLS + half * W4_A_SUB);
            if (nsub == W4_SUB) {
                uint32_t cols[64];
#pragma unroll
                for (int u = 0; u < W4_SUB; ++u)
                    w4_unpack_row<DT>(prow + u * sub_stride, cols + 32 * u);
                tmem_st64(a_dst, cols);
            } else {
                uint32_t cols[32];
                w4_unpack_row<DT>(prow, cols);
                tmem_st32(a_dst, cols);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(cfull(cb));
            ++step;
            if (++stage == W4_STAGES) {
                stage = 0;
                phase ^= 1u;
            }
            if (++cb == W4_CONVS) {
                cb = 0;
                cph ^= 1u;
            }
        }
    } else {
        // ------------------------------- epilogue -------------------------------
        // thread (lane quarter q, lane) holds output channel n0 + 32 q + lane
        // (and, in stage 2, n0 + 128 + 32 q + lane) for every row of the block
        const int q = warp & 3;
        const int ch = q * 32 + lane;
        int local = 0, rslot = 0;
        uint32_t rphase = 0;
        for (;;) {
            int got = 1, tl = -1;
            if (lane == 0) {
                got = mbar_wait_bounded(tidf(rslot), rphase, abort_flag, p.err) ? 1 : 0;
                if (got) {
                    tl = tid_ring[rslot];
                    mbar_arrive(tide(rslot));
                }
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            tl = __shfl_sync(0xffffffffu, tl, 0);
            if (++rslot == W4_TRING) {
                rslot = 0;
                rphase ^= 1u;
            }
            if (!got || tl < 0) break;
            const W4Tile ti = w4_tile(p, list, blk_g, blk_m, blk_rows, n_blocks, tl);
            const bool gu = ti.phase == 0;
            const int N = gu ? p.d_e : p.d_h;
            OutT *out = reinterpret_cast<OutT *>(gu ? p.h : p.y);
            const int acc = local & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
            int ready = 1;
            if (lane == 0) ready = mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, p.err) ? 1 : 0;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * W4_ACC_COLS);
            int np = (ti.rows + 15) & ~15;
            if (np > W4_TOK_ROWS) np = W4_TOK_ROWS;
            const int rows = ti.rows < np ? ti.rows : np;
            const int f0 = ti.n0 + ch;
            const int f1 = gu ? -1 : ti.n0 + 128 + ch;
            if (p.out_i32) {
                // W4A8: the fp32 sums hold integers of magnitude <= 2^24 (a K
                // chunk is at most 16384 long), so the conversion is exact.
                // Transposed results (Ct[n, m], 8 or more rows) go through a
                // per-warp shared-memory transpose so that each store or atomic
                // instruction covers runs of 16 consecutive m.
                const bool xposed = p.ld_row == 1 && p.ld_col >= 8;
                int *xt = xpose + (warp - 2) * (32 * 17);
#pragma unroll 1
                for (int j0 = 0; j0 < np; j0 += 16) {
                    uint32_t a[16], b[16];
                    tmem_ld16(t_row + j0, a);
                    tmem_ld16(t_row + np + j0, b);
                    tmem_ld_wait();
                    if (xposed) {
#pragma unroll
                        for (int hsel = 0; hsel < 2; ++hsel) {
                            __syncwarp();
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                xt[lane * 17 + jj] = __float2int_rn(__uint_as_float(hsel ? b[jj] : a[jj]));
                            __syncwarp();
                            const int jj = lane & 15, j = j0 + jj;
#pragma unroll 4
                            for (int i = 0; i < 16; ++i) {
                                const int c = 2 * i + (lane >> 4);  // channel within the warp's 32
                                const int n = ti.n0 + hsel * 128 + q * 32 + c;
                                if (j < rows && n < N) {
                                    int32_t *o = p.out_i32 + (ti.m_start + j) + static_cast<int64_t>(n) * p.ld_col;
                                    const int v = xt[c * 17 + jj];
                                    if (p.atomic_out)
                                        atomicAdd(o, v);
                                    else
                                        *o = v;
                                }
                            }
                        }
                        continue;
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        if (j < rows) {
                            const int64_t m = ti.m_start + j;
                            int32_t *o0 = p.out_i32 + m * p.ld_row + static_cast<int64_t>(f0) * p.ld_col;
                            int32_t *o1 = p.out_i32 + m * p.ld_row + static_cast<int64_t>(f1) * p.ld_col;
                            const int v0 = __float2int_rn(__uint_as_float(a[jj]));
                            const int v1 = __float2int_rn(__uint_as_float(b[jj]));
                            if (p.atomic_out) {
                                if (f0 < N) atomicAdd(o0, v0);
                                if (f1 < N) atomicAdd(o1, v1);
                            } else {
                                if (f0 < N) *o0 = v0;
                                if (f1 < N) *o1 = v1;
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty(acc));
                ++local;
                continue;
            }
            // per-channel scales (1 when absent): stage 1 gate / up, stage 2 the two channels
            float sa = 1.0f, sb = 1.0f;
            if (gu) {
                if (f0 < N && p.s_gate) sa = __ldg(p.s_gate + static_cast<int64_t>(ti.g) * N + f0);
                if (f0 < N && p.s_up) sb = __ldg(p.s_up + static_cast<int64_t>(ti.g) * N + f0);
            } else if (p.s_down) {
                if (f0 < N) sa = __ldg(p.s_down + static_cast<int64_t>(ti.g) * N + f0);
                if (f1 < N) sb = __ldg(p.s_down + static_cast<int64_t>(ti.g) * N + f1);
            }
#pragma unroll 1
            for (int j0 = 0; j0 < np; j0 += 16) {
                uint32_t a[16], b[16];
                tmem_ld16(t_row + j0, a);
                tmem_ld16(t_row + np + j0, b);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = j0 + jj;
                    if (j < rows) {
                        const int64_t r = static_cast<int64_t>(ti.m_start + j) * N;
                        if (gu) {
                            const float gv = __uint_as_float(a[jj]) * sa;
                            const float sv = gv * __frcp_rn(1.0f + __expf(-gv));
                            if (f0 < N) out[r + f0] = from_f32<OutT>(sv * (__uint_as_float(b[jj]) * sb));
                        } else {
                            const float rwj = p.row_weights ? __ldg(p.row_weights + ti.m_start + j) : 1.0f;
                            if (f0 < N) out[r + f0] = from_f32<OutT>((__uint_as_float(a[jj]) * sa) * rwj);
                            if (f1 < N) out[r + f1] = from_f32<OutT>((__uint_as_float(b[jj]) * sb) * rwj);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(acc));
            if (gu) {
                // this warp's h rows are stored: count them for the stage-2 tiles
                __threadfence();
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) counter_publish(p.ready + ti.bx);
            }
            ++local;
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, W4_TMEM_COLS);
    }
}

template <int DT>
cudaError_t launch_w4_typed(const CUtensorMap *maps, const W4Params &p, int grid, cudaStream_t stream) {
    auto kern = grouped_mlp_w4_kernel<DT>;
    static std::atomic<bool> attr_done[64];  // zero-initialised; several host threads may launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, W4_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    return launch_pdl(kern, dim3(grid), dim3(W4_THREADS), W4_SMEM_BYTES, stream, maps[0], maps[1], p);
}

}  // namespace

int64_t pack_int4_bytes(int64_t E, int64_t N, int64_t K, int R) {
    if (E <= 0 || N <= 0 || K <= 0 || K % W4_BK != 0 || R <= 0) return -1;
    return E * ((N + R - 1) / R) * R * (K / 2);
}

cudaError_t launch_pack_int4(const uint8_t *plain, int64_t E, int64_t N, int64_t K, int R, uint8_t *packed,
                             cudaStream_t stream) {
    const int64_t n_words = pack_int4_bytes(E, N, K, R) / 4;
    if (n_words <= 0) return cudaSuccess;
    const int64_t blocks = (n_words + 255) / 256;
    return launch_pdl(pack_int4_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                      reinterpret_cast<const uint32_t *>(plain), E, N, K, R, reinterpret_cast<uint32_t *>(packed));
}

cudaError_t launch_grouped_mlp_w4(int dtype, const void *x, const int32_t *gather_idx, int64_t T,
                                  const uint8_t *q_gate, const uint8_t *q_up, const uint8_t *q_down,
                                  const float *s_gate, const float *s_up, const float *s_down,
                                  const int32_t *sizes, const int32_t *offsets,
                                  const int32_t *padded, const int32_t *gidx, int64_t m_blocks,
                                  const float *row_weights, int64_t n_rows, int64_t d_h,
                                  int64_t d_e, int64_t E, void *h, void *y, int32_t *ready,
                                  int32_t *err, cudaStream_t stream) {
    if (n_rows <= 0 || m_blocks <= 0) return cudaSuccess;
    if (m_blocks > W4_MAX_BLOCKS) return cudaErrorInvalidValue;
    const int t16 = dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap maps[2];
    const uint64_t uh = static_cast<uint64_t>(d_h), ue = static_cast<uint64_t>(d_e);
    {   // x [T, d_h], one row per box (four rows per gather)
        const uint64_t dims[2] = {uh, static_cast<uint64_t>(T)}, st[1] = {uh * 2};
        const uint32_t box[2] = {W4_BK, 1};
        if (!encode_tma_map(&maps[0], t16, 2, x, dims, st, box, 1)) return cudaErrorInvalidValue;
    }
    {   // h [n_rows, d_e], 64 rows per box
        const uint64_t dims[2] = {ue, static_cast<uint64_t>(n_rows)}, st[1] = {ue * 2};
        const uint32_t box[2] = {W4_BK, W4_TOK_ROWS};
        if (!encode_tma_map(&maps[1], t16, 2, h, dims, st, box, 1)) return cudaErrorInvalidValue;
    }
    W4Params p{};
    p.sizes = sizes;
    p.offsets = offsets;
    p.padded = padded;
    p.gidx = gidx;
    p.gather_idx = gather_idx;
    p.q_gate = q_gate;
    p.q_up = q_up;
    p.q_down = q_down;
    p.row_weights = row_weights;
    p.s_gate = s_gate;
    p.s_up = s_up;
    p.s_down = s_down;
    p.ready = ready;
    p.tile_counter = ready + m_blocks;
    p.h = h;
    p.y = y;
    p.m_blocks = static_cast<int>(m_blocks);
    p.d_h = static_cast<int>(d_h);
    p.d_e = static_cast<int>(d_e);
    p.nt0 = static_cast<int>((d_e + 127) / 128);
    p.nt1 = static_cast<int>((d_h + 255) / 256);
    p.kb0 = static_cast<int>(d_h / W4_BK);
    p.kb1 = static_cast<int>(d_e / W4_BK);
    p.err = err;
    p.ksplit = 1;
    p.kchunk = p.kb1;
    const int64_t tiles = m_blocks * (p.nt0 + p.nt1);
    const int grid = mlp_grid(tiles);
    if (dtype == kBF16) return launch_w4_typed<kBF16>(maps, p, grid, stream);
    return launch_w4_typed<kF16>(maps, p, grid, stream);
}

namespace {

// W4A8 activations: int8 rows (row r = x[idx[r]], or x[r] without idx) ->
// fp16 rows; every int8 value is exact in fp16.  A row index outside
// [0, T) is reported on err and its row written as zeros.
__global__ void w4a8_rows_kernel(const int8_t *__restrict__ x, const int32_t *__restrict__ idx, int64_t T,
                                 int64_t n_rows, int64_t K, __half *__restrict__ out, int32_t *err,
                                 int32_t *zero_a, int64_t n_a, int32_t *zero_b, int64_t n_b) {
    griddep_wait();
    griddep_launch_dependents();
    // the GEMM's counters and, when it adds K chunks, its output start at zero
    const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = tid; i < n_a; i += nthr) zero_a[i] = 0;
    for (int64_t i = tid; i < n_b; i += nthr) zero_b[i] = 0;
    const int64_t per_row = K / 16;
    const int64_t total = n_rows * per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / per_row, c = i - r * per_row;
        const int64_t src = idx ? __ldg(idx + r) : r;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (src >= 0 && src < T) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + src * K) + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t h[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __half2 a = __halves2half2(__int2half_rn(static_cast<int8_t>(w[q] & 0xFFu)),
                                                 __int2half_rn(static_cast<int8_t>((w[q] >> 8) & 0xFFu)));
                const __half2 b = __halves2half2(__int2half_rn(static_cast<int8_t>((w[q] >> 16) & 0xFFu)),
                                                 __int2half_rn(static_cast<int8_t>(w[q] >> 24)));
                h[2 * q] = *reinterpret_cast<const uint32_t *>(&a);
                h[2 * q + 1] = *reinterpret_cast<const uint32_t *>(&b);
            }
            lo = make_uint4(h[0], h[1], h[2], h[3]);
            hi = make_uint4(h[4], h[5], h[6], h[7]);
        } else if (err && c == 0) {
            atomicExch(err, kErrDeviceFlag);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(out + r * K) + 2 * c;
        dst[0] = lo;
        dst[1] = hi;
    }
}

// ---------------------------------------------------------------------------
// W4A8 with few rows (the dense form, M <= GV_MAX_M): a weight-streaming GEMV
// on the CUDA cores.  With so few rows per weight the work is the weight
// bytes, and unpacking into tensor memory costs more than the MMAs save.  A
// CTA owns one 256-channel tile and a K range: a producer warp streams the
// tile's packed sub-steps (8 KB each, contiguous) into a ring of shared
// memory with bulk copies, so the bytes in flight are bounded by shared
// memory rather than registers, and each consumer thread owns one output
// channel.  Each 32-bit word holds 8 weights as value + 8 in the tiled
// layout's nibble order (elements 0, 2, 4, 6 in nibbles 0-3, 1, 3, 5, 7 in
// 4-7), so one AND gives the bytes of elements (0, 4, 1, 5) and a shift and
// AND those of (2, 6, 3, 7); dp4a multiplies them with the activation bytes
// staged in the same order: sum_k a_k w_k = sum_k a_k (w_k + 8) - 8 sum_k a_k,
// exact in int32.
// ---------------------------------------------------------------------------
constexpr int GV_THREADS = 256;             // consumers: the tile's channels
constexpr int GV_BLOCK = GV_THREADS + 32;   // + the producer warp
constexpr int GV_MAX_M = 8;
constexpr int GV_MAX_SUB = 64;              // 64-wide sub-steps of a CTA's K range
constexpr int GV_RING = 12;                 // stages of the weight ring
constexpr int GV_STAGE = GV_THREADS * 32;   // one sub-step of the tile, 8 KB

__host__ __device__ constexpr int gv_smem_bytes(int mt) {
    return GV_RING * GV_STAGE + 2 * mt * GV_MAX_SUB * 8 * 4 + 2 * GV_RING * 8 + mt * 4 + 16;
}

template <int MT>
__global__ void __launch_bounds__(GV_BLOCK)
    w4a8_gemv_kernel(const int8_t *__restrict__ A, int M, const uint8_t *__restrict__ B, int N, int K,
                     int kchunk, int32_t *__restrict__ Ct, int atomic_out, int32_t *err) {
    extern __shared__ __align__(128) uint8_t gv_smem[];
    uint8_t *ring = gv_smem;
    uint32_t *a_lo = reinterpret_cast<uint32_t *>(ring + GV_RING * GV_STAGE);  // [MT][GV_MAX_SUB * 8]
    uint32_t *a_hi = a_lo + MT * GV_MAX_SUB * 8;
    uint64_t *bars = reinterpret_cast<uint64_t *>(a_hi + MT * GV_MAX_SUB * 8);  // full, empty
    int *a_sum = reinterpret_cast<int *>(bars + 2 * GV_RING);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(a_sum + MT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int i) { return bar0 + 8u * i; };
    auto empty_bar = [&](int i) { return bar0 + 8u * (GV_RING + i); };
    const int kb = K / W4_BK;
    const int s0 = blockIdx.y * kchunk;
    const int ns = min(kchunk, kb - s0);
    if (ns <= 0) return;  // the whole CTA
    if (threadIdx.x == 0) {
        for (int i = 0; i < GV_RING; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), GV_THREADS / 32);  // one arrival per consumer warp
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < MT) a_sum[threadIdx.x] = 0;
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();

    if (warp == GV_THREADS / 32) {
        // ------------------------------ producer ------------------------------
        const uint8_t *src = B + (static_cast<int64_t>(blockIdx.x) * kb + s0) * GV_STAGE;
        if (lane == 0) {
            for (int s = 0; s < ns; ++s) {
                const int st = s % GV_RING;
                if (s >= GV_RING &&
                    !mbar_wait_bounded(empty_bar(st), static_cast<uint32_t>((s / GV_RING) & 1) ^ 1u, abort_flag, err))
                    break;
                mbar_arrive_expect_tx(full_bar(st), GV_STAGE);
                w4_bulk_g2s(smem_u32(ring + st * GV_STAGE), src + static_cast<int64_t>(s) * GV_STAGE, GV_STAGE,
                            full_bar(st), l2_policy_evict_first());
            }
        }
        return;
    }
    // ------------------------------ consumers ------------------------------
    // the CTA's activations, 8 elements per word pair, in the weight words' byte order
    const int groups = ns * 8;
    for (int m = 0; m < M; ++m) {
        int part = 0;
        for (int g = threadIdx.x; g < groups; g += GV_THREADS) {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(A + static_cast<int64_t>(m) * K +
                                                                  static_cast<int64_t>(s0) * W4_BK) + g);
            a_lo[m * GV_MAX_SUB * 8 + g] = __byte_perm(v.x, v.y, 0x5140);  // elements 0, 4, 1, 5
            a_hi[m * GV_MAX_SUB * 8 + g] = __byte_perm(v.x, v.y, 0x7362);  // elements 2, 6, 3, 7
            part = __dp4a(static_cast<int>(v.x), 0x01010101, part);
            part = __dp4a(static_cast<int>(v.y), 0x01010101, part);
        }
#pragma unroll
        for (int sh = 16; sh >= 1; sh >>= 1) part += __shfl_xor_sync(0xffffffffu, part, sh);
        if (lane == 0) atomicAdd(&a_sum[m], part);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(GV_THREADS) : "memory");  // consumers only
    const int t = threadIdx.x;
    // the two 16-byte halves of this channel's 32 bytes, read in a lane-dependent
    // order so that the eight lanes of an access phase hit eight bank groups
    const int sel = (lane >> 2) & 1;
    int acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0;
    bool ok = true;
    for (int s = 0; s < ns; ++s) {
        const int st = s % GV_RING;
        if (!mbar_wait_bounded(full_bar(st), static_cast<uint32_t>((s / GV_RING) & 1), abort_flag, err)) {
            ok = false;
            break;
        }
        const uint4 *r = reinterpret_cast<const uint4 *>(ring + st * GV_STAGE + t * 32);
        const uint4 x0 = r[sel], x1 = r[sel ^ 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(st));
        const uint4 w0 = sel ? x1 : x0, w1 = sel ? x0 : x1;
        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int lo = static_cast<int>(wv[q] & 0x0F0F0F0Fu);
            const int hi = static_cast<int>((wv[q] >> 4) & 0x0F0F0F0Fu);
            const int g = s * 8 + q;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < M) {
                    acc[m] = __dp4a(lo, static_cast<int>(a_lo[m * GV_MAX_SUB * 8 + g]), acc[m]);
                    acc[m] = __dp4a(hi, static_cast<int>(a_hi[m * GV_MAX_SUB * 8 + g]), acc[m]);
                }
            }
        }
    }
    if (!ok) {
        // after a timeout, let the copies still in flight land before the CTA exits
        for (int s = 0; s < ns && s < GV_RING; ++s) {
            const int last = s + ((ns - 1 - s) / GV_RING) * GV_RING;  // the last use of stage s
            w4_wait_drain(full_bar(s), static_cast<uint32_t>((last / GV_RING) & 1));
        }
        return;
    }
    const int n = blockIdx.x * GV_THREADS + t;
    if (n < N) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const int v = acc[m] - 8 * a_sum[m];
                int32_t *o = Ct + static_cast<int64_t>(n) * M + m;
                if (atomic_out)
                    atomicAdd(o, v);
                else
                    *o = v;
            }
        }
    }
}

template <int MT>
cudaError_t launch_gemv_typed(const int8_t *A, int M, const uint8_t *B, int64_t N, int64_t K, int32_t *Ct,
                              int32_t *err, cudaStream_t stream) {
    const int64_t kb = K / W4_BK, nt = (N + GV_THREADS - 1) / GV_THREADS;
    constexpr int smem = gv_smem_bytes(MT);
    static_assert(smem <= 232448, "shared memory per CTA");
    // about one wave at two CTAs per SM (one where two do not fit), at most
    // GV_MAX_SUB sub-steps each
    const int per_sm = 2 * smem <= 232448 ? 2 : 1;
    int64_t ks = std::max<int64_t>(1, per_sm * device_sm_count() / nt);
    const int64_t kchunk = std::min<int64_t>(GV_MAX_SUB, std::max<int64_t>(1, (kb + ks - 1) / ks));
    ks = (kb + kchunk - 1) / kchunk;
    if (ks > 65535 || nt > 0x7fffffff) return cudaErrorInvalidValue;
    static std::atomic<bool> attr_done[64];  // zero-initialised; several host threads may launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        const cudaError_t e =
            cudaFuncSetAttribute(w4a8_gemv_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    if (ks > 1) {
        const cudaError_t e = cudaMemsetAsync(Ct, 0, static_cast<size_t>(N * M) * 4, stream);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(w4a8_gemv_kernel<MT>, dim3(static_cast<unsigned>(nt), static_cast<unsigned>(ks)),
                      dim3(GV_BLOCK), smem, stream, A, M, B, static_cast<int>(N), static_cast<int>(K),
                      static_cast<int>(kchunk), Ct, ks > 1 ? 1 : 0, err);
}

}  // namespace

W4a8Plan w4a8_plan(int64_t blocks, int64_t N, int64_t K) {
    W4a8Plan pl;
    const int64_t kb = K / W4_BK, nt = (N + 255) / 256;
    // split K until the grid is about one tile per SM, in chunks of at least
    // four sub-steps, and in any case into chunks of at most 256 sub-steps
    // (16384 products: the fp32 sums stay integers of magnitude <= 2^24)
    int64_t ks = device_sm_count() / std::max<int64_t>(1, blocks * nt);
    ks = std::min<int64_t>(ks, std::max<int64_t>(1, kb / 4));
    ks = std::max<int64_t>(ks, (kb + kW4a8MaxChunkSub - 1) / kW4a8MaxChunkSub);
    ks = std::max<int64_t>(ks, 1);
    pl.kchunk = (kb + ks - 1) / ks;
    pl.ksplit = (kb + pl.kchunk - 1) / pl.kchunk;
    return pl;
}

cudaError_t launch_gemm_w4a8(const int8_t *x, const int32_t *gather_idx, int64_t T, const uint8_t *B,
                             const int32_t *sizes, const int32_t *offsets, const int32_t *padded,
                             const int32_t *gidx, int64_t m_blocks, int64_t dense_rows, int64_t n_rows,
                             int64_t N, int64_t K, void *rows_f16, int32_t *counters, int32_t *out,
                             int64_t ld_row, int64_t ld_col, int64_t out_elems, int32_t *err,
                             cudaStream_t stream) {
    if (n_rows <= 0 || N <= 0) return cudaSuccess;
    if (dense_rows <= 0 && (m_blocks <= 0 || m_blocks > W4_MAX_BLOCKS)) return cudaErrorInvalidValue;
    if (dense_rows > W4_TOK_ROWS || K % W4_BK != 0) return cudaErrorInvalidValue;
    if (dense_rows > 0 && dense_rows <= GV_MAX_M && ld_row == 1 && ld_col == dense_rows) {
        // few rows: the CUDA-core GEMV (Ct [N, M])
        const int M = static_cast<int>(dense_rows);
        if (M == 1) return launch_gemv_typed<1>(x, M, B, N, K, out, err, stream);
        if (M == 2) return launch_gemv_typed<2>(x, M, B, N, K, out, err, stream);
        if (M <= 4) return launch_gemv_typed<4>(x, M, B, N, K, out, err, stream);
        return launch_gemv_typed<8>(x, M, B, N, K, out, err, stream);
    }
    const int64_t blocks = dense_rows > 0 ? 1 : m_blocks;
    const W4a8Plan pl = w4a8_plan(blocks, N, K);
    {
        const int64_t work = std::max<int64_t>(n_rows * (K / 16), pl.ksplit > 1 ? out_elems : 0);
        const int64_t nb = std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, 4LL * device_sm_count()));
        const cudaError_t e = launch_pdl(w4a8_rows_kernel, dim3(static_cast<unsigned>(nb)), dim3(256), 0, stream,
                                         x, gather_idx, T, n_rows, K, static_cast<__half *>(rows_f16), err,
                                         counters, blocks + 1, out, pl.ksplit > 1 ? out_elems : int64_t(0));
        if (e != cudaSuccess) return e;
    }
    CUtensorMap maps[2];
    {   // the fp16 rows [n_rows, K], 64 rows per box (both map slots: stage-1 rows are unused)
        const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(n_rows)},
                       st[1] = {static_cast<uint64_t>(K) * 2};
        const uint32_t box[2] = {W4_BK, W4_TOK_ROWS};
        if (!encode_tma_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, rows_f16, dims, st, box, 1))
            return cudaErrorInvalidValue;
        maps[0] = maps[1];
    }
    W4Params p{};
    p.sizes = sizes;
    p.offsets = offsets;
    p.padded = padded;
    p.gidx = gidx;
    p.q_down = B;
    p.ready = counters;
    p.tile_counter = counters + blocks;
    p.h = rows_f16;
    p.m_blocks = static_cast<int>(blocks);
    p.d_h = static_cast<int>(N);
    p.d_e = static_cast<int>(K);
    p.nt0 = 0;
    p.nt1 = static_cast<int>((N + 255) / 256);
    p.kb0 = 0;
    p.kb1 = static_cast<int>(K / W4_BK);
    p.err = err;
    p.ksplit = static_cast<int>(pl.ksplit);
    p.kchunk = static_cast<int>(pl.kchunk);
    p.dense_rows = static_cast<int>(dense_rows);
    p.out_i32 = out;
    p.ld_row = ld_row;
    p.ld_col = ld_col;
    p.atomic_out = pl.ksplit > 1 ? 1 : 0;
    const int grid = mlp_grid(blocks * p.nt1 * pl.ksplit);
    return launch_w4_typed<kF16>(maps, p, grid, stream);
}

}  // namespace moe

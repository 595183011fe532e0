// grouped_gemm_w4.cu -- the expert MLP (both GEMM stages in one launch) with
// int4 weights and 16-bit activations (weight-only W4A16), for up to 64
// tokens, where the expert weights are read once per step and their bytes
// are the whole cost.
//
// Weight format (TileLang tutorial ch.18 skeletons.py, w4a8_dequant_gemm):
// int4 values two per byte, element j of a row in byte j/2 at nibble j%2
// from the low end, two's complement; the kernel unpacks them on chip and
// casts them to the compute type before the GEMM (the module notes: the same
// kernel with 16-bit activations is the weight-only W4A16 form).  Reading: an
// optional fp32 scale per output channel multiplies the fp32 sum.
//
// launch_pack_int4 moves each 32-bit word of that format (8 elements) into
// the order the converter wants -- elements 2m and 2m+1 in nibbles m and
// m+4 -- stored offset-binary (value + 8), so that one AND-OR with the fp16
// (or bf16) exponent of 1024 (128) and one packed subtraction of 1032 (136)
// give two exact values.
//
// Kernel (one persistent CTA per SM, 320 threads):
//   warp 0      producer: per 64-wide K step, one stage of a 9-deep ring:
//               the block's rows (stage 1: up to 64 token rows gathered from
//               x by four-row TMA gathers; stage 2: 64 rows of h) and the
//               packed weights of 256 output channels (8 KB);
//   warps 6..9  converters: unpack the stage's 256 x 64 weights into one of
//               two 32 KB tiles in the 128-byte swizzled K-major layout the
//               tensor cores read (the layout TMA gives 16-bit weights);
//   warp 1      MMA: tcgen05.mma M=128 N=rows (two per K=16 step: weight
//               halves as the M operand, the block's rows as N) into a TMEM
//               accumulator, double buffered;
//   warps 2..5  epilogue: scales, silu(gate)*up for stage 1, row-masked
//               stores; a stage-1 warp-tile publishes its h rows on the
//               block's counter for the stage-2 tiles.
// Tiles are taken as in the 16-bit expert MLP: CTA b starts with tile b,
// the rest come from a shared counter; stage-2 tiles wait (bounded) for
// their block's h.  Every wait is bounded; on a timeout the kernel records
// MOE_ERR_TIMEOUT, lets its copies and MMAs land, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int W4_BK = 64;                        // K elements per step
constexpr int W4_ROWS = 256;                     // weight rows (output channels) per tile
constexpr int W4_PACK_ROW = W4_BK / 2;           // 32 packed bytes per row and step
constexpr int W4_PACK_BYTES = W4_ROWS * W4_PACK_ROW;  // 8 KB
constexpr int W4_TOK_ROWS = 64;                  // the most rows a block may hold here
constexpr int W4_TOK_BYTES = W4_TOK_ROWS * W4_BK * 2;  // 8 KB, 128-byte swizzled
constexpr int W4_STAGE_BYTES = W4_TOK_BYTES + W4_PACK_BYTES;
constexpr int W4_STAGES = 9;
constexpr int W4_CONV_BYTES = W4_ROWS * W4_BK * 2;  // 32 KB, two 16 KB MMA operands
constexpr int W4_CONVS = 2;
constexpr int W4_THREADS = 320;
constexpr int W4_CONV_WARP0 = 6;                 // converter warps 6..9
constexpr int W4_CONV_WARPS = 4;
constexpr int W4_EPI_WARPS = 4;
constexpr int W4_TRING = 4;
constexpr int W4_ACC_COLS = 128;                 // 2 x up to 64 columns per accumulator
constexpr int W4_TMEM_COLS = 256;
constexpr int W4_MAX_BLOCKS = 1088;              // M blocks the schedule lists
constexpr int W4_BAR_BYTES = 512;
constexpr int W4_SCHED_BYTES = W4_MAX_BLOCKS * (4 * 3 + 1) + 64 * 4;
constexpr int W4_SMEM_BYTES = 1024 + W4_CONVS * W4_CONV_BYTES + W4_STAGES * W4_STAGE_BYTES +
                              W4_BAR_BYTES + W4_SCHED_BYTES;
static_assert(W4_SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(W4_STAGE_BYTES % 1024 == 0 && W4_CONV_BYTES % 1024 == 0, "swizzle atoms");

// ---------------------------------------------------------------------------
// repack: one thread per 32-bit word (8 elements)
// ---------------------------------------------------------------------------
__global__ void pack_int4_kernel(const uint32_t *__restrict__ plain, int64_t n_words,
                                 uint32_t *__restrict__ packed) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n_words) return;
    const uint32_t w = plain[i];
    uint32_t o = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t nib = (w >> (4 * e)) & 0xFu;
        const int slot = (e & 1) ? 4 + (e >> 1) : (e >> 1);
        o |= nib << (4 * slot);
    }
    packed[i] = o ^ 0x88888888u;  // offset-binary: value + 8
}

struct W4Params {
    const int32_t *sizes, *offsets, *padded, *gidx;
    const int32_t *gather_idx;  // stage-1 rows: token indices into x
    const float *row_weights;
    const float *s_gate, *s_up, *s_down;
    int *ready;         // per M block: stage-1 epilogue warp-tiles stored
    int *tile_counter;  // next tile beyond the first wave
    void *h, *y;
    int m_blocks, d_h, d_e;
    int nt0, nt1;       // output tiles per block: stage 1 (128 columns), stage 2 (256)
    int kb0, kb1;       // K steps: stage 1 (d_h / 64), stage 2 (d_e / 64)
    int *err;
};

struct W4Tile {
    int g, m_start, rows, n0, bx, phase;
};

// Tile t of the launch: the stage-1 tiles of every listed block first, then
// the stage-2 tiles in the same block order.
__device__ __forceinline__ W4Tile w4_tile(const W4Params &p, const int *list, const int *blk_g,
                                          const int *blk_m, const uint8_t *blk_rows, int n_blocks,
                                          int t) {
    W4Tile ti;
    const int n0_tiles = n_blocks * p.nt0;
    int pos, nt;
    if (t < n0_tiles) {
        ti.phase = 0;
        pos = t / p.nt0;
        nt = t - pos * p.nt0;
        ti.n0 = nt * 128;
    } else {
        ti.phase = 1;
        t -= n0_tiles;
        pos = t / p.nt1;
        nt = t - pos * p.nt1;
        ti.n0 = nt * 256;
    }
    const int bx = list[pos];
    ti.bx = bx;
    ti.g = blk_g[bx];
    ti.m_start = blk_m[bx];
    ti.rows = blk_rows[bx];
    return ti;
}

__device__ __forceinline__ void w4_wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long start = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - start > kWaitTimeoutNs) return;
}

// Unpack one 32-bit word (8 elements, the repacked layout) into 8 values of
// the compute type, in element order.
template <int DT>
__device__ __forceinline__ uint4 w4_unpack8(uint32_t w) {
    constexpr uint32_t MAGIC = DT == kBF16 ? 0x43004300u : 0x64006400u;  // 128 / 1024, twice
    uint32_t q[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) q[m] = ((w >> (4 * m)) & 0x000F000Fu) | MAGIC;
    uint4 r;
    if (DT == kBF16) {
        const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
        __nv_bfloat162 v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&q[m]), off);
        r = make_uint4(*reinterpret_cast<uint32_t *>(&v[0]), *reinterpret_cast<uint32_t *>(&v[1]),
                       *reinterpret_cast<uint32_t *>(&v[2]), *reinterpret_cast<uint32_t *>(&v[3]));
    } else {
        const __half2 off = __floats2half2_rn(1032.0f, 1032.0f);
        __half2 v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = __hsub2(*reinterpret_cast<__half2 *>(&q[m]), off);
        r = make_uint4(*reinterpret_cast<uint32_t *>(&v[0]), *reinterpret_cast<uint32_t *>(&v[1]),
                       *reinterpret_cast<uint32_t *>(&v[2]), *reinterpret_cast<uint32_t *>(&v[3]));
    }
    return r;
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
                          const __grid_constant__ CUtensorMap tmQg,   // [E, d_e, d_h/2] u8, box 32 x 128
                          const __grid_constant__ CUtensorMap tmQu,
                          const __grid_constant__ CUtensorMap tmQd,   // [E, d_h, d_e/2] u8, box 32 x 256
                          const W4Params p) {
    using OutT = typename Elem<DT>::T;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *conv = smem;                                      // [W4_CONVS][32 KB]
    uint8_t *stages = conv + W4_CONVS * W4_CONV_BYTES;          // [W4_STAGES][tokens 8 KB | packed 8 KB]
    uint64_t *bars = reinterpret_cast<uint64_t *>(stages + W4_STAGES * W4_STAGE_BYTES);
    // barriers: pfull, pempty [stages]; cfull, cempty [convs]; tfull, tempty [2]; tidf, tide [ring]
    constexpr int NBARS = 2 * W4_STAGES + 2 * W4_CONVS + 4 + 2 * W4_TRING;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *tid_ring = reinterpret_cast<int *>(tmem_slot + 2);
    volatile int *stage_flag = reinterpret_cast<volatile int *>(tid_ring + W4_TRING);  // 1 = K step, 0 = end
    static_assert(NBARS * 8 + 8 + 4 * W4_TRING + 4 * W4_STAGES <= W4_BAR_BYTES, "barrier area");
    int *list = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + W4_BAR_BYTES);
    int *blk_g = list + W4_MAX_BLOCKS;
    int *blk_m = blk_g + W4_MAX_BLOCKS;
    uint8_t *blk_rows = reinterpret_cast<uint8_t *>(blk_m + W4_MAX_BLOCKS);
    int *scan_scratch = reinterpret_cast<int *>(blk_rows + W4_MAX_BLOCKS);
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
            mbar_init(pempty(s), W4_CONV_WARPS + 1);  // every converter warp and the MMA's commit
        }
        for (int c = 0; c < W4_CONVS; ++c) {
            mbar_init(cfull(c), W4_CONV_WARPS);
            mbar_init(cempty(c), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull(a), 1);
            mbar_init(tempty(a), W4_EPI_WARPS);
        }
        for (int i = 0; i < W4_TRING; ++i) {
            mbar_init(tidf(i), 1);
            mbar_init(tide(i), 1 + W4_EPI_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmH);
        tma_prefetch_desc(&tmQg);
        tma_prefetch_desc(&tmQu);
        tma_prefetch_desc(&tmQd);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), W4_TMEM_COLS);
        tmem_relinquish();
    }
    griddep_wait();  // the tables, x and the counters come from earlier kernels
    griddep_launch_dependents();

    // ----- schedule: the non-empty M blocks in order, with their lookups -----
    int n_blocks = 0;
    {
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
            mine += rows > 0;
        }
        int base = w4_cta_scan(mine, scan_scratch, &n_blocks);
        for (int bx = lo; bx < hi; ++bx)
            if (blk_rows[bx] > 0) list[base++] = bx;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = n_blocks * (p.nt0 + p.nt1);

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t pol_first = l2_policy_evict_first();  // weights are read once
            int stage = 0;
            uint32_t phase = 0;
            long issued = 0;
            bool ok = true;
            int rslot = 0;
            uint32_t rphase = 0;
            int next_tile = static_cast<int>(gridDim.x) + atomicAdd(p.tile_counter, 1);
            for (int it = 0; ok; ++it) {
                int tile = it == 0 ? static_cast<int>(blockIdx.x) : next_tile;
                if (it > 0) next_tile = static_cast<int>(gridDim.x) + atomicAdd(p.tile_counter, 1);
                if (tile >= total) tile = -1;
                if (!mbar_wait_bounded(tide(rslot), rphase ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tid_ring[rslot] = tile;
                mbar_arrive(tidf(rslot));
                if (++rslot == W4_TRING) {
                    rslot = 0;
                    rphase ^= 1u;
                }
                if (tile < 0) break;
                const W4Tile ti = w4_tile(p, list, blk_g, blk_m, blk_rows, n_blocks, tile);
                // stage 2 reads its block's h rows: all stage-1 warp-tiles stored
                if (ti.phase == 1 &&
                    !counter_wait_bounded(p.ready + ti.bx, W4_EPI_WARPS * p.nt0, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                int np = (ti.rows + 15) & ~15;
                if (np > W4_TOK_ROWS) {  // the host admits at most 64 tokens
                    np = W4_TOK_ROWS;
                    if (p.err) atomicExch(p.err, kErrDeviceFlag);
                }
                const int kblocks = ti.phase == 0 ? p.kb0 : p.kb1;
                const uint32_t tx = static_cast<uint32_t>((ti.phase == 0 ? np * W4_BK * 2 : W4_TOK_BYTES) +
                                                          W4_PACK_BYTES);
                const int32_t *ids = p.gather_idx + ti.m_start;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(pempty(stage), phase ^ 1u, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = stages + stage * W4_STAGE_BYTES;
                    const uint32_t tok = smem_u32(st), pk = smem_u32(st + W4_TOK_BYTES);
                    const uint32_t fb = pfull(stage);
                    stage_flag[stage] = 1;
                    mbar_arrive_expect_tx(fb, tx);
                    if (ti.phase == 0) {
                        // four token rows per copy; rows past the block repeat its first row
                        for (int r = 0; r < np; r += 4) {
                            const int i0 = __ldg(ids + (r < ti.rows ? r : 0));
                            const int i1 = __ldg(ids + (r + 1 < ti.rows ? r + 1 : 0));
                            const int i2 = __ldg(ids + (r + 2 < ti.rows ? r + 2 : 0));
                            const int i3 = __ldg(ids + (r + 3 < ti.rows ? r + 3 : 0));
                            tma_gather4(tok + static_cast<uint32_t>(r * W4_BK * 2), &tmX, fb, kb * W4_BK, i0, i1,
                                        i2, i3);
                        }
                        tma_load_3d_hint(pk, &tmQg, fb, kb * W4_PACK_ROW, ti.n0, ti.g, pol_first);
                        tma_load_3d_hint(pk + W4_PACK_BYTES / 2, &tmQu, fb, kb * W4_PACK_ROW, ti.n0, ti.g,
                                         pol_first);
                    } else {
                        tma_load_2d(tok, &tmH, fb, kb * W4_BK, ti.m_start);
                        tma_load_3d_hint(pk, &tmQd, fb, kb * W4_PACK_ROW, ti.n0, ti.g, pol_first);
                    }
                    ++issued;
                    if (++stage == W4_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
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
    } else if (warp == 1) {
        // --------------------------------- MMA ---------------------------------
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
                const int kblocks = ti.phase == 0 ? p.kb0 : p.kb1;
                const int acc = local & 1;
                const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
                if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * W4_ACC_COLS);
                int np = (ti.rows + 15) & ~15;
                if (np > W4_TOK_ROWS) np = W4_TOK_ROWS;
                const uint32_t idesc = idesc_f16(DT == kBF16, 128, static_cast<uint32_t>(np));
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(cfull(cb), cph, abort_flag, p.err) ||
                        !mbar_wait_bounded(pfull(stage), phase, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t cvb = smem_u32(conv + cb * W4_CONV_BYTES);
                    const uint64_t a0 = smem_desc_sw128(cvb);
                    const uint64_t a1 = smem_desc_sw128(cvb + W4_CONV_BYTES / 2);
                    const uint64_t bd = smem_desc_sw128(smem_u32(stages + stage * W4_STAGE_BYTES));
#pragma unroll
                    for (int k = 0; k < W4_BK / 16; ++k) {
                        const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
                        // D[channel][row]: first 128 channels into columns [0, np), the rest into [np, 2np)
                        tc_mma_f16(d_tmem, a0 + 2u * k, bd + 2u * k, idesc, accum);
                        tc_mma_f16(d_tmem + static_cast<uint32_t>(np), a1 + 2u * k, bd + 2u * k, idesc, accum);
                    }
                    tc_commit(pempty(stage));  // the rows' stage may be refilled once these finish
                    tc_commit(cempty(cb));     // and the unpacked weights overwritten
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
    } else if (warp >= W4_CONV_WARP0) {
        // ------------------------------ converters ------------------------------
        // warp cw unpacks rows 16 i + 4 cw + lane / 8 (i = 0..15) of every
        // stage: lane reads one 32-bit word (8 weights) and writes 16 bytes at
        // the swizzled position (chunk ^ row % 8) of the row
        const int cw = warp - W4_CONV_WARP0;
        const int chunk = lane & 7;
        int stage = 0, cb = 0;
        uint32_t phase = 0, cph = 0;
        for (;;) {
            if (!mbar_wait_bounded(pfull(stage), phase, abort_flag, p.err)) break;
            if (stage_flag[stage] == 0) break;
            if (!mbar_wait_bounded(cempty(cb), cph ^ 1u, abort_flag, p.err)) break;
            const uint8_t *pk = stages + stage * W4_STAGE_BYTES + W4_TOK_BYTES;
            uint8_t *cv = conv + cb * W4_CONV_BYTES;
#pragma unroll 4
            for (int i = 0; i < W4_ROWS / (4 * W4_CONV_WARPS); ++i) {
                const int row = i * (4 * W4_CONV_WARPS) + cw * 4 + (lane >> 3);
                const uint32_t w = *reinterpret_cast<const uint32_t *>(pk + row * W4_PACK_ROW + chunk * 4);
                *reinterpret_cast<uint4 *>(cv + row * (W4_BK * 2) + ((chunk ^ (row & 7)) << 4)) =
                    w4_unpack8<DT>(w);
            }
            // the tensor cores read the tile through the async proxy
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(cfull(cb));
                mbar_arrive(pempty(stage));
            }
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
    static bool attr_done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, W4_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    return launch_pdl(kern, dim3(grid), dim3(W4_THREADS), W4_SMEM_BYTES, stream, maps[0], maps[1],
                      maps[2], maps[3], maps[4], p);
}

}  // namespace

cudaError_t launch_pack_int4(const uint8_t *plain, int64_t n_bytes, uint8_t *packed,
                             cudaStream_t stream) {
    if (n_bytes <= 0) return cudaSuccess;
    const int64_t n_words = n_bytes / 4;
    const int64_t blocks = (n_words + 255) / 256;
    return launch_pdl(pack_int4_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                      reinterpret_cast<const uint32_t *>(plain), n_words, reinterpret_cast<uint32_t *>(packed));
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
    const int t8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUtensorMap maps[5];
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
    {   // packed W_gate / W_up [E, d_e, d_h / 2] bytes, 128 channels per box
        const uint64_t dims[3] = {uh / 2, ue, static_cast<uint64_t>(E)}, st[2] = {uh / 2, ue * uh / 2};
        const uint32_t box[3] = {W4_PACK_ROW, 128, 1};
        if (!encode_tma_map(&maps[2], t8, 3, q_gate, dims, st, box, 0) ||
            !encode_tma_map(&maps[3], t8, 3, q_up, dims, st, box, 0))
            return cudaErrorInvalidValue;
    }
    {   // packed W_down [E, d_h, d_e / 2] bytes, 256 channels per box
        const uint64_t dims[3] = {ue / 2, uh, static_cast<uint64_t>(E)}, st[2] = {ue / 2, uh * ue / 2};
        const uint32_t box[3] = {W4_PACK_ROW, 256, 1};
        if (!encode_tma_map(&maps[4], t8, 3, q_down, dims, st, box, 0)) return cudaErrorInvalidValue;
    }
    W4Params p{};
    p.sizes = sizes;
    p.offsets = offsets;
    p.padded = padded;
    p.gidx = gidx;
    p.gather_idx = gather_idx;
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
    const int64_t tiles = m_blocks * (p.nt0 + p.nt1);
    const int grid = static_cast<int>(tiles < device_sm_count() ? tiles : device_sm_count());
    if (dtype == kBF16) return launch_w4_typed<kBF16>(maps, p, grid, stream);
    return launch_w4_typed<kF16>(maps, p, grid, stream);
}

}  // namespace moe

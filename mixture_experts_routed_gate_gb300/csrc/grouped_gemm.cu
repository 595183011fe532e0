// grouped_gemm.cu -- the two grouped expert GEMMs of the routed MoE forward on
// the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// Stage 1 (CSDN "tilelang kernel stage 1 gate+up"; skeletons.py moe_routed_kernel):
//   h[rows of block bx] = silu(A W_gate[g]^T) * (A W_up[g]^T)
// Stage 2 (CSDN "tilelang kernel stage 2 down"):
//   y[rows of block bx] = (h W_down[g]^T) (* row weight)
// with the block -> (expert g, first row m_start, valid rows) lookup of the
// pages' dispatch contract.
//
// Design (one persistent CTA per SM, 224 threads):
//   warp 0      TMA producer: per 64-wide K step loads the 128-row A tile and the
//               256-row B tile (stage 1: 128 W_gate rows + 128 W_up rows of the
//               same output columns; stage 2: 256 W_down rows) into a 4-deep
//               shared-memory ring, 128-byte swizzled.
//   warp 1      MMA issuer: one thread issues tcgen05.mma M=128 N=256 K=16 into
//               a TMEM accumulator (2 x 256 columns, double buffered so the
//               epilogue of tile i overlaps the main loop of tile i+1).  Blocks
//               with at most 64 valid rows are computed swapped: two M=128
//               MMAs with the weight halves as A and the block's rows as B
//               (N = rows rounded up to 16), a fraction of the tensor work.
//   warp 6      second MMA issuer: a swapped tile's second MMA of each pair
//               (one thread issues a small-N MMA only about every 85 cycles).
//   warps 2..5  epilogue: tcgen05.ld the accumulator (thread = row), stage 1
//               fuses silu(gate)*up, stage 2 the optional row weight; round to
//               the activation dtype and store only the block's valid rows.
// Tiles are (M block, N tile) pairs; the blocks are ordered by the schedule
// below (full and partial blocks interleaved; blocks with no valid rows, the
// padding blocks the tables create, left out).  The single-stage modes deal
// them round-robin to the CTAs; the expert MLP mode hands out every tile from
// a shared counter, in order, each CTA taking its next tile two K steps
// before it issues the current one's last copy.
//
// The expert MLP mode runs both stages in one launch: the stage-1 tiles come
// first in the tile order, then the stage-2 tiles in the same block order.
// Each epilogue warp that stores part of a block's h publishes it on a
// per-block counter; the producer starts a stage-2 tile once its block's
// counter is complete.  Tiles are taken in order and every stage-1 tile
// precedes every stage-2 tile, so when a stage-2 tile is taken, the stage-1
// tiles it waits on have all been taken by running CTAs, whose own progress
// waits on nothing later: every wait ends, whether or not the whole grid is
// resident at once.
// Both stages then share one wave tail and no launch gap separates them.
//
// Every wait is bounded (see
// mbar_wait_bounded): on a timeout the kernel records kErrTimeout, drains the
// copies and MMAs it issued, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 x 2 B = 128 B: one swizzle span per row
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int NUM_THREADS = 224;  // 7 warps: producer, MMA, 4 epilogue, second MMA issuer
constexpr int MMA2_WARP = 6;
constexpr int MMA_N = 256;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int B_BYTES = MMA_N * BK * 2;      // 32 KB
constexpr int BAR_BYTES = 256;
// Tile ids handed from the producer to the MMA and epilogue warps when tiles
// are taken from a global counter (expert MLP mode).
constexpr int TRING = 4;
// The producer takes its next tile from the shared counter this many K steps
// before the end of the current tile (see the producer)
constexpr int NEXT_FETCH = 2;
// K steps of the first tile prefetched into L2 before the dependency wait
// (few-token launches; 16 x 32 KB per CTA, about 78 MB over the grid)
constexpr int PREFETCH_STEPS = 16;
// Blocks with at most this many valid rows run "swapped": the weight tile is
// the M=128 operand and the block's rows the N operand (N = rows rounded up
// to 16), so a mostly-padding block costs N/128 of a full MMA.
constexpr int SWAP_MAX_ROWS = 64;
constexpr int MAX_SCHED = 1024;  // M blocks the in-kernel schedule can order
// block list; per block: expert, first row, valid rows, class; per listed
// full block: run start / length (int16); scan scratch
constexpr int SCHED_BYTES = MAX_SCHED * 4 * 3 + 2 * MAX_SCHED * 2 + 2 * MAX_SCHED + 64;

// MODE_MLP: both stages in one launch.  MODE_MLP_FEW: the same when every
// block holds at most 64 rows (rows gathered from at most 64 tokens): a ring
// stage then needs 64 rows of A, so five stages fit and each SM keeps 160 KB
// of weights in flight instead of 128 KB.
enum { MODE_GATE_UP = 0, MODE_DOWN = 1, MODE_MLP = 2, MODE_MLP_FEW = 3 };

template <int MODE>
struct Layout {
    static constexpr bool MLP = MODE == MODE_MLP || MODE == MODE_MLP_FEW;
    static constexpr int NST = MODE == MODE_MLP_FEW ? 5 : STAGES;
    static constexpr int A_SLOT = MODE == MODE_MLP_FEW ? SWAP_MAX_ROWS * BK * 2 : A_BYTES;
    static constexpr int SMEM = 1024 /*alignment slack*/ + NST * (A_SLOT + B_BYTES) + BAR_BYTES + SCHED_BYTES;
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

struct PhaseParams {
    void *out;     // h (stage 1) or y (stage 2), row-major [rows, N]
    int n_tiles;   // output tiles per M block
    int k_blocks;  // 64-wide K steps
    int N;         // output columns
};

struct GemmParams {
    const int32_t *sizes;
    const int32_t *offsets;
    const int32_t *padded;
    const int32_t *gidx;
    const float *row_weights;
    int *ready;  // MODE_MLP: per M block, stage-1 epilogue warp-tiles stored
    int *tile_counter;  // MODE_MLP: next tile to take (null: fixed round-robin)
    // MODE_MLP: stage 1 gathers its rows straight from the tokens x (through
    // tmX) by these indices (null: stage 1 reads the gathered rows through tmA0)
    const int32_t *gather_idx;
    PhaseParams ph[2];  // [0] stage 1 (gate/up), [1] stage 2 (down)
    int m_blocks;
    int *err;
    // MODE_MLP, every expert at most one block (a few tokens): the expert
    // count, for the start-up prefetch below (0: none)
    int prefetch_experts;
};

struct TileInfo {
    int g, m_start, rows, n0, bx, phase;
    bool big;  // part of a large expert's stripe-major run
};

constexpr int EPI_WARPS = 4;

// Valid rows of M block bx (the pages' actual_rows) and its first row.
__device__ __forceinline__ int block_rows(const GemmParams &p, int bx, int *g_out, int *m_start) {
    const int g = __ldg(p.gidx + bx);
    const int rel = bx * BM - __ldg(p.padded + g);
    int rows = __ldg(p.sizes + g) - rel;
    rows = rows < 0 ? 0 : (rows > BM ? BM : rows);
    if (g_out) *g_out = g;
    if (m_start) *m_start = rel + __ldg(p.offsets + g);
    return rows;
}

// The tile schedule.  Non-empty M blocks are split by expert size: blocks of
// experts with at least 128 rows (their full blocks are tensor-bound) and
// the single block of each smaller expert (mostly padding: streaming the
// expert's weights is the limit).  Small experts' tiles go block by block.
// Large experts' tiles go expert by expert, and inside an expert N-stripe
// first: every block of the expert on weight stripe n before stripe n+1, so
// a stripe is fetched from HBM once while the expert's activation rows are
// re-read from L2.  The two tile sequences are interleaved evenly,
// so every window of tiles dealt round-robin to the persistent CTAs mixes
// both kinds and the tensor pipe and HBM are busy at the same time.
struct Schedule {
    const int *list;       // [n_full full blocks][n_partial partial blocks]; null = natural order
    const int16_t *run_start;  // per full block: index of its expert's first full block in list
    const int16_t *run_len;    // per full block: number of full blocks of its expert
    const int *blk_g;          // per M block: expert, first row, valid rows (from the tables)
    const int *blk_m;
    const uint8_t *blk_rows;
    int n_full, n_blocks;
};

__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, const Schedule &sc, int tile,
                                              int n_tiles, int out_n) {
    int bx, nt;
    bool tile_is_big = false;
    if (sc.list) {
        const int64_t n_full_t = static_cast<int64_t>(sc.n_full) * n_tiles;
        const int64_t n_all_t = static_cast<int64_t>(sc.n_blocks) * n_tiles;
        const int64_t hb = tile * n_full_t / n_all_t;         // full tiles before position tile
        const int64_t hn = (tile + 1) * n_full_t / n_all_t;
        if (hn > hb) {
            tile_is_big = true;
            const int fb = static_cast<int>(hb / n_tiles);  // full block whose run holds it
            const int rs = sc.run_start[fb], rl = sc.run_len[fb];
            const int64_t o = hb - static_cast<int64_t>(rs) * n_tiles;
            nt = static_cast<int>(o / rl);
            bx = sc.list[rs + static_cast<int>(o - static_cast<int64_t>(nt) * rl)];
        } else {
            const int64_t lt = tile - hb;                     // partial tile index
            bx = sc.list[sc.n_full + static_cast<int>(lt / n_tiles)];
            nt = static_cast<int>(lt % n_tiles);
        }
    } else {
        bx = tile / n_tiles;
        nt = tile - bx * n_tiles;
    }
    TileInfo t;
    if (sc.list) {
        t.g = sc.blk_g[bx];
        t.m_start = sc.blk_m[bx];
        t.rows = sc.blk_rows[bx];
    } else {
        t.rows = block_rows(p, bx, &t.g, &t.m_start);
    }
    t.n0 = nt * out_n;
    t.bx = bx;
    t.phase = 0;
    t.big = sc.list != nullptr && tile_is_big;
    return t;
}

// The parameters of stage `phase` (field by field: indexing the kernel
// parameter array with a run-time index would copy it to local memory).
__device__ __forceinline__ PhaseParams phase_params_of(const GemmParams &p, int phase) {
    PhaseParams r;
    r.out = phase == 0 ? p.ph[0].out : p.ph[1].out;
    r.n_tiles = phase == 0 ? p.ph[0].n_tiles : p.ph[1].n_tiles;
    r.k_blocks = phase == 0 ? p.ph[0].k_blocks : p.ph[1].k_blocks;
    r.N = phase == 0 ? p.ph[0].N : p.ph[1].N;
    return r;
}

// Tile `tile` of the launch: its stage and its place in that stage's order.
// n0_tiles = stage-1 tiles of the launch (MODE_MLP only).
template <int MODE>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams &p, const Schedule &sc, int tile,
                                                int n0_tiles) {
    int phase = MODE == MODE_DOWN ? 1 : 0;
    if (Layout<MODE>::MLP && tile >= n0_tiles) {
        phase = 1;
        tile -= n0_tiles;
    }
    TileInfo t = tile_info(p, sc, tile, phase == 0 ? p.ph[0].n_tiles : p.ph[1].n_tiles,
                           phase == 0 ? 128 : 256);
    t.phase = phase;
    return t;
}

// Exclusive scan of one int per thread across the CTA; returns the total.
template <int NT>
__device__ __forceinline__ int cta_exclusive_scan(int v, int *scratch, int *total) {
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
    for (int w = 0; w < NT / 32; ++w) {
        const int x = scratch[w];
        if (w < warp) base += x;
        tot += x;
    }
    __syncthreads();
    *total = tot;
    return base + incl - v;
}

// A wait used only while winding down after an abort: bounded, ignores the
// abort flag (the point is to let in-flight hardware work land).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
    unsigned long long start = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - start > kWaitTimeoutNs) return;
    }
}

// An epilogue warp has stored its part of a stage-1 tile: make the stores
// visible at gpu scope (and to the async proxy that TMA reads through), then
// count the warp-tile on the block's counter.
__device__ __forceinline__ void publish_h(int *ctr, int lane) {
    __threadfence();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (lane == 0) counter_publish(ctr);
}

// Stage 1 reads rows A through tmA0 (or gathers token rows through tmX) and
// W_gate / W_up through tmB0 / tmB1; stage 2 reads h through tmA1 and W_down
// through tmB2.
template <int DT, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB2,
                        const __grid_constant__ CUtensorMap tmX, const GemmParams p) {
    constexpr bool HAS0 = MODE != MODE_DOWN, HAS1 = MODE != MODE_GATE_UP;
    constexpr bool IS_MLP = Layout<MODE>::MLP;
    constexpr int NST = Layout<MODE>::NST, A_SLOT = Layout<MODE>::A_SLOT;
    constexpr uint32_t IDESC = idesc_f16(DT == kBF16, BM, MMA_N);
    using OutT = typename Elem<DT>::T;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + NST * A_SLOT;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + NST * B_BYTES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * NST + 4 + 2 * TRING);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *tid_ring = reinterpret_cast<int *>(tmem_slot + 2);
    static_assert((2 * NST + 4 + 2 * TRING) * 8 + 8 + 4 * TRING <= BAR_BYTES, "barrier area");
    int *sched = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + BAR_BYTES);
    int *blk_g = sched + MAX_SCHED;
    int *blk_m = blk_g + MAX_SCHED;
    int16_t *sched_rs = reinterpret_cast<int16_t *>(blk_m + MAX_SCHED);
    int16_t *sched_rl = sched_rs + MAX_SCHED;
    uint8_t *sched_cls = reinterpret_cast<uint8_t *>(sched_rl + MAX_SCHED);
    uint8_t *blk_rows = sched_cls + MAX_SCHED;
    int *sched_scratch = reinterpret_cast<int *>(blk_rows + MAX_SCHED);
    static_assert(MAX_SCHED % 4 == 0, "scratch alignment");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (NST + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * NST + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * NST + 2 + a); };
    auto tidf_bar = [&](int i) { return bar0 + 8u * (2 * NST + 4 + i); };
    auto tide_bar = [&](int i) { return bar0 + 8u * (2 * NST + 4 + TRING + i); };
    // tiles from the global counter (in order, each CTA taking the next one
    // when its producer is ready) instead of a fixed round-robin deal
    const bool dynamic = IS_MLP && p.tile_counter != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 2);  // the commits of the two MMA threads
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 2);  // the commits of the two MMA threads
            mbar_init(tempty_bar(a), 4);  // one arrival per epilogue warp
        }
        for (int i = 0; i < TRING; ++i) {
            mbar_init(tidf_bar(i), 1);
            mbar_init(tide_bar(i), 2 + EPI_WARPS);  // both MMA threads and every epilogue warp
        }
        *abort_flag = 0;
        fence_mbar_init();
        if (HAS0) {
            tma_prefetch_desc(&tmA0);
            tma_prefetch_desc(&tmB0);
            tma_prefetch_desc(&tmB1);
        }
        if (HAS1) {
            tma_prefetch_desc(&tmA1);
            tma_prefetch_desc(&tmB2);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    // everything above is independent of the previous kernel; the tables and
    // rows below are not
    // While the routing kernels still run, pull the first K steps of this
    // CTA's first tile into L2.  With one block per expert and every expert
    // routed, stage-1 tile b (CTA b's first) is stripe b % n_tiles of expert
    // b / n_tiles; when some expert is idle the guess is off by a few stripes,
    // which other CTAs read soon after.  Weights do not come from the
    // routing, so this may run before the dependency wait.
    if (IS_MLP && p.prefetch_experts > 0 && warp == 0 && lane == 0) {
        const int nt = p.ph[0].n_tiles;
        const int g = static_cast<int>(blockIdx.x) / nt;
        if (g < p.prefetch_experts) {
            const int n0 = (static_cast<int>(blockIdx.x) - g * nt) * 128;
            for (int kb = 0; kb < PREFETCH_STEPS && kb < p.ph[0].k_blocks; ++kb) {
                tma_prefetch_3d(&tmB0, kb * BK, n0, g);
                tma_prefetch_3d(&tmB1, kb * BK, n0, g);
            }
        }
    }
    griddep_wait();
    griddep_launch_dependents();
    // dynamic: the first tile comes from the shared counter too (claimed here,
    // its round trip hidden behind the schedule build), so every tile a CTA
    // waits on belongs to a CTA that is already running
    int first_tile = 0;
    if (dynamic && threadIdx.x == 0) first_tile = atomicAdd(p.tile_counter, 1);
    // ----- schedule: classify the M blocks, list full and partial ones -----
    Schedule sc{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0, p.m_blocks};
    if (p.m_blocks <= MAX_SCHED) {
        for (int bx = threadIdx.x; bx < p.m_blocks; bx += NUM_THREADS) {
            int g, m0;
            const int r = block_rows(p, bx, &g, &m0);
            blk_g[bx] = g;
            blk_m[bx] = m0;
            blk_rows[bx] = static_cast<uint8_t>(r);
            // every block of an expert with at least one full block joins that
            // expert's run (its tail too: one sweep over the expert's weights)
            sched_cls[bx] = r == 0 ? 0 : (__ldg(p.sizes + g) >= BM ? 2 : 1);
        }
        __syncthreads();
        const int chunk = (p.m_blocks + NUM_THREADS - 1) / NUM_THREADS;
        const int lo = threadIdx.x * chunk;
        const int hi = min(p.m_blocks, lo + chunk);
        int nf = 0, np = 0;
        for (int bx = lo; bx < hi; ++bx) {
            nf += sched_cls[bx] == 2;
            np += sched_cls[bx] == 1;
        }
        int tot_f, tot_p;
        int bf = cta_exclusive_scan<NUM_THREADS>(nf, sched_scratch, &tot_f);
        int bpart = cta_exclusive_scan<NUM_THREADS>(np, sched_scratch, &tot_p);
        for (int bx = lo; bx < hi; ++bx) {
            if (sched_cls[bx] == 2) sched[bf++] = bx;
            else if (sched_cls[bx] == 1) sched[tot_f + bpart++] = bx;
        }
        __syncthreads();
        // runs of full blocks of one expert (consecutive in the list, block
        // order = expert order): each full block learns its run's start/length
        for (int i = threadIdx.x; i < tot_f; i += NUM_THREADS) {
            const int g = blk_g[sched[i]];
            int lo_i = i, hi_i = i;
            while (lo_i > 0 && blk_g[sched[lo_i - 1]] == g) --lo_i;
            while (hi_i + 1 < tot_f && blk_g[sched[hi_i + 1]] == g) ++hi_i;
            sched_rs[i] = static_cast<int16_t>(lo_i);
            sched_rl[i] = static_cast<int16_t>(hi_i - lo_i + 1);
        }
        sc.list = sched;
        sc.run_start = sched_rs;
        sc.run_len = sched_rl;
        sc.blk_g = blk_g;
        sc.blk_m = blk_m;
        sc.blk_rows = blk_rows;
        sc.n_full = tot_f;
        sc.n_blocks = tot_f + tot_p;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n0_tiles = HAS0 ? sc.n_blocks * p.ph[0].n_tiles : 0;
    const int total = n0_tiles + (HAS1 ? sc.n_blocks * p.ph[1].n_tiles : 0);

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        // the whole warp: lane 0 takes tiles, arms the stage barriers and issues
        // the weight (and tiled row) copies; when stage-1 rows are gathered from
        // x, lane j holds the token ids of rows 4j .. 4j+3 for the tile and
        // issues their gather every K step (128 rows for a full tile)
        const uint64_t pol_first = l2_policy_evict_first();
        const uint64_t pol_last = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        long issued = 0;
        bool ok = true;
        int rslot = 0;
        uint32_t rphase = 0;
        // dynamic: every tile, the first included, comes from the shared
        // counter, in order, so a stage-2 tile is only ever taken after all
        // stage-1 tiles (which precede it in the order) were taken by running
        // CTAs: progress does not depend on all CTAs being resident at once.
        // The next tile is taken NEXT_FETCH K steps before the current tile's
        // last copy is issued: late enough that at the end of the launch the
        // last tiles go to CTAs that are about to be free (taking it at the
        // start of the current tile bound them a whole tile early), early
        // enough that the atomic's round trip is hidden (its result is first
        // used at the next tile).
        int next_tile = first_tile;
        bool have_next = true;
        for (int it = 0; ok; ++it) {
            int tile = blockIdx.x + it * static_cast<int>(gridDim.x);
            if (dynamic) {
                // pass the tile id on (-1: none left)
                int go = 1;
                if (lane == 0) {
                    if (!have_next) next_tile = atomicAdd(p.tile_counter, 1);
                    tile = next_tile;
                    have_next = false;
                    if (tile >= total) tile = -1;
                    go = mbar_wait_bounded(tide_bar(rslot), rphase ^ 1u, abort_flag, p.err) ? 1 : 0;
                    if (go) {
                        tid_ring[rslot] = tile;
                        mbar_arrive(tidf_bar(rslot));
                    }
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                tile = __shfl_sync(0xffffffffu, tile, 0);
                if (++rslot == TRING) {
                    rslot = 0;
                    rphase ^= 1u;
                }
                if (!go) {
                    ok = false;
                    break;
                }
                if (tile < 0) break;
            } else if (tile >= total) {
                break;
            }
            const TileInfo ti = decode_tile<MODE>(p, sc, tile, n0_tiles);
            if (ti.rows == 0) continue;
            // a stage-2 tile reads h rows of its block: wait until every
            // stage-1 epilogue warp-tile of the block has stored them
            if (IS_MLP && ti.phase == 1) {
                int go = 1;
                if (lane == 0)
                    go = counter_wait_bounded(p.ready + ti.bx, EPI_WARPS * p.ph[0].n_tiles, abort_flag, p.err) ? 1
                                                                                                                 : 0;
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
            }
            const int kblocks = phase_params_of(p, ti.phase).k_blocks;
            // stage-1 rows gathered from x: the block's rows rounded up to 4, one
            // four-row gather per producer lane.  The MMA reads np (swapped) or 128
            // rows of the slot; the ones past the gathered rows hold stale bytes
            // that only reach accumulator rows / columns nobody stores, and every
            // copy saved shortens the producer's issue path, which paces a K step
            const bool gather = IS_MLP && ti.phase == 0 && p.gather_idx != nullptr;
            const int nrow_g = (ti.rows + 3) & ~3;
            const uint32_t stage_tx = static_cast<uint32_t>((gather ? nrow_g * BK * 2 : A_SLOT) + B_BYTES);
            // this lane's four token ids (rows past the block repeat its first row)
            int i0 = 0, i1 = 0, i2 = 0, i3 = 0;
            const bool gatherer = gather && 4 * lane < nrow_g;
            if (gatherer) {
                const int32_t *ids = p.gather_idx + ti.m_start;
                const int r = 4 * lane;
                i0 = __ldg(ids + (r < ti.rows ? r : 0));
                i1 = __ldg(ids + (r + 1 < ti.rows ? r + 1 : 0));
                i2 = __ldg(ids + (r + 2 < ti.rows ? r + 2 : 0));
                i3 = __ldg(ids + (r + 3 < ti.rows ? r + 3 : 0));
            }
            const int fetch_kb = kblocks > NEXT_FETCH ? kblocks - NEXT_FETCH : 0;
            for (int kb = 0; kb < kblocks; ++kb) {
                if (dynamic && lane == 0 && kb == fetch_kb) {
                    next_tile = atomicAdd(p.tile_counter, 1);
                    have_next = true;
                }
                int go = 1;
                if (lane == 0) go = mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.err) ? 1 : 0;
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
                const uint32_t fb = full_bar(stage);
                const uint32_t a_dst = smem_u32(sA + stage * A_SLOT);
                const uint32_t b_dst = smem_u32(sB + stage * B_BYTES);
                if (lane == 0) mbar_arrive_expect_tx(fb, stage_tx);
                __syncwarp();  // the stage's byte count is armed before any copy lands
                if (gather) {
                    // x rows are read by k experts and every N tile of a block: keep them
                    if (gatherer)
                        tma_gather4_hint(a_dst + static_cast<uint32_t>(4 * lane * BK * 2), &tmX, fb, kb * BK, i0,
                                         i1, i2, i3, pol_last);
                } else if (lane == 0) {
                    // a large expert's rows and weight stripes are reused by the
                    // tiles of its run: keep them; a small expert's weights are
                    // read by one block only: let them leave L2 first
                    const CUtensorMap *ta = HAS0 && ti.phase == 0 ? &tmA0 : &tmA1;
                    if (ti.big) tma_load_2d_hint(a_dst, ta, fb, kb * BK, ti.m_start, pol_last);
                    else tma_load_2d(a_dst, ta, fb, kb * BK, ti.m_start);
                }
                if (lane == 0) {
                    const uint64_t polb = ti.big ? pol_last : pol_first;
                    if (HAS0 && ti.phase == 0) {
                        tma_load_3d_hint(b_dst, &tmB0, fb, kb * BK, ti.n0, ti.g, polb);
                        tma_load_3d_hint(b_dst + B_BYTES / 2, &tmB1, fb, kb * BK, ti.n0, ti.g, polb);
                    } else {
                        tma_load_3d_hint(b_dst, &tmB2, fb, kb * BK, ti.n0, ti.g, polb);
                    }
                }
                ++issued;
                if (++stage == NST) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            // let every copy still in flight land before shared memory goes away
            for (long j = 1; j <= NST && j <= issued; ++j) {
                const long i = issued - j;
                mbar_wait_drain(full_bar(static_cast<int>(i % NST)), static_cast<uint32_t>((i / NST) & 1));
            }
        }
    } else if (warp == 1 || warp == MMA2_WARP) {
        // ------------------------------- MMA issuers --------------------------------
        // One thread issues a small-N MMA about every 85 cycles, so a swapped
        // tile's two accumulators are issued by two threads: warp 1 the first
        // (and every MMA of an unswapped tile), warp 6 the second, each in the
        // K order one thread would use (the results do not change).  Both wait
        // for every stage and commit it.
        const bool mma_b = warp == MMA2_WARP;
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            uint32_t last_bar = 0, last_parity = 0;
            bool committed = false;
            int rslot = 0;
            uint32_t rphase = 0;
            for (int it = 0; ok; ++it) {
                int tile = blockIdx.x + it * static_cast<int>(gridDim.x);
                if (dynamic) {
                    if (!mbar_wait_bounded(tidf_bar(rslot), rphase, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tile = tid_ring[rslot];
                    mbar_arrive(tide_bar(rslot));
                    if (++rslot == TRING) {
                        rslot = 0;
                        rphase ^= 1u;
                    }
                    if (tile < 0) break;
                } else if (tile >= total) {
                    break;
                }
                const TileInfo ti = decode_tile<MODE>(p, sc, tile, n0_tiles);
                if (ti.rows == 0) continue;
                const int kblocks = phase_params_of(p, ti.phase).k_blocks;
                const int acc = local & 1;
                const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
                if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
                const bool swap = ti.rows <= SWAP_MAX_ROWS;
                const int np = (ti.rows + 15) & ~15;
                const uint32_t idesc_sw = idesc_f16(DT == kBF16, BM, static_cast<uint32_t>(np));
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = smem_desc_sw128(smem_u32(sA + stage * A_SLOT));
                    const uint64_t b_desc = smem_desc_sw128(smem_u32(sB + stage * B_BYTES));
                    if (swap) {
                        // D[feature][row]: first 128 weight rows into columns [0, np)
                        // (warp 1), the other 128 into [np, 2np) (warp 6)
                        const uint64_t wb_desc =
                            mma_b ? smem_desc_sw128(smem_u32(sB + stage * B_BYTES + B_BYTES / 2)) : b_desc;
                        const uint32_t d_acc = mma_b ? d_tmem + static_cast<uint32_t>(np) : d_tmem;
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            tc_mma_f16(d_acc, wb_desc + 2u * k, a_desc + 2u * k, idesc_sw, (kb | k) != 0 ? 1u : 0u);
                    } else if (!mma_b) {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            // +32 bytes per K=16 step inside the 128-byte swizzled row
                            tc_mma_f16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, IDESC,
                                       (kb | k) != 0 ? 1u : 0u);
                        }
                    }
                    tc_commit(empty_bar(stage));  // frees the smem stage when these MMAs finish
                    last_bar = empty_bar(stage);
                    last_parity = phase;
                    committed = true;
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(tfull_bar(acc));  // accumulator ready for the epilogue
                ++local;
            }
            if (!ok && committed) mbar_wait_drain(last_bar, last_parity);
        }
    } else {
        // --------------------------------- epilogue ---------------------------------
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        const int row = q * 32 + lane;
        int local = 0;
        int rslot = 0;
        uint32_t rphase = 0;
        for (int it = 0;; ++it) {
            int tile = blockIdx.x + it * static_cast<int>(gridDim.x);
            if (dynamic) {
                // lane 0 takes the id (one arrival per warp), the warp follows
                int got = 1, tl = -1;
                if (lane == 0) {
                    got = mbar_wait_bounded(tidf_bar(rslot), rphase, abort_flag, p.err) ? 1 : 0;
                    if (got) {
                        tl = tid_ring[rslot];
                        mbar_arrive(tide_bar(rslot));
                    }
                }
                got = __shfl_sync(0xffffffffu, got, 0);
                tl = __shfl_sync(0xffffffffu, tl, 0);
                if (++rslot == TRING) {
                    rslot = 0;
                    rphase ^= 1u;
                }
                if (!got || tl < 0) break;
                tile = tl;
            } else if (tile >= total) {
                break;
            }
            const TileInfo ti = decode_tile<MODE>(p, sc, tile, n0_tiles);
            if (ti.rows == 0) continue;
            const bool gu = HAS0 && ti.phase == 0;  // stage 1: silu(gate) * up
            const int out_cols = gu ? 128 : 256;
            const PhaseParams php = phase_params_of(p, ti.phase);
            const int N = php.N;
            OutT *const out_base = reinterpret_cast<OutT *>(php.out);
            const int acc = local & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
            // one lane waits, the warp reconverges before the .sync.aligned TMEM loads
            int ready = 1;
            if (lane == 0) ready = mbar_wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.err) ? 1 : 0;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * ACC_COLS);
            if (ti.rows <= SWAP_MAX_ROWS) {
                // swapped tile: this thread holds output feature `row` (and, for
                // stage 2, feature 128 + row) for every row j of the block
                const int np = (ti.rows + 15) & ~15;
                OutT *out = out_base;
                const int f0 = ti.n0 + row;
                const int f1 = gu ? -1 : ti.n0 + 128 + row;
#pragma unroll 1
                for (int j0 = 0; j0 < np; j0 += 16) {
                    uint32_t a[16], b[16];
                    tmem_ld16(t_row + j0, a);
                    tmem_ld16(t_row + np + j0, b);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        if (j < ti.rows) {
                            const int64_t r = static_cast<int64_t>(ti.m_start + j) * N;
                            if (gu) {
                                const float gv = __uint_as_float(a[jj]);
                                const float s = gv * __frcp_rn(1.0f + __expf(-gv));
                                if (f0 < N) out[r + f0] = from_f32<OutT>(s * __uint_as_float(b[jj]));
                            } else {
                                const float rwj = p.row_weights ? __ldg(p.row_weights + ti.m_start + j) : 1.0f;
                                if (f0 < N) out[r + f0] = from_f32<OutT>(__uint_as_float(a[jj]) * rwj);
                                if (f1 < N) out[r + f1] = from_f32<OutT>(__uint_as_float(b[jj]) * rwj);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
                if (IS_MLP && gu) publish_h(p.ready + ti.bx, lane);
                ++local;
                continue;
            }
            const bool valid = row < ti.rows;
            OutT *out_row = out_base + static_cast<int64_t>(ti.m_start + (valid ? row : 0)) * N;
            float rw = 1.0f;
            if (!gu && p.row_weights != nullptr && valid) rw = __ldg(p.row_weights + ti.m_start + row);
#pragma unroll 1
            for (int c = 0; c < out_cols / 16; ++c) {
                const int col = ti.n0 + c * 16;
                uint32_t packed[8];
                if (gu) {
                    uint32_t g[16], u[16];
                    tmem_ld16(t_row + c * 16, g);
                    tmem_ld16(t_row + 128 + c * 16, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float v[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const float gv = __uint_as_float(g[2 * i + h]);
                            const float uv = __uint_as_float(u[2 * i + h]);
                            const float s = gv * __frcp_rn(1.0f + __expf(-gv));
                            v[h] = s * uv;
                        }
                        packed[i] = pack2<DT>(v[0], v[1]);
                    }
                } else {
                    uint32_t r[16];
                    tmem_ld16(t_row + c * 16, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        packed[i] = pack2<DT>(__uint_as_float(r[2 * i]) * rw,
                                              __uint_as_float(r[2 * i + 1]) * rw);
                }
                if (valid && col < N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(out_row + col);
                    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (IS_MLP && gu) publish_h(p.ready + ti.bx, lane);
            ++local;
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    // looked up once (a function-local static: thread-safe initialisation)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return nullptr;
    }();
    return fn;
}

}  // namespace

// Any tensor map: dims / strides (bytes, dims 1..rank-1) / box, innermost first.
bool encode_tma_map(CUtensorMap *m, int data_type, int rank, const void *ptr, const uint64_t *dims,
                    const uint64_t *strides_bytes, const uint32_t *box, int swizzle_128b) {
    auto fn = encode_fn();
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    CUresult r = fn(m, static_cast<CUtensorMapDataType>(data_type), static_cast<cuuint32_t>(rank),
                    const_cast<void *>(ptr), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle_128b ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major [rows, inner] 16-bit matrix, box = box_inner x box_rows, no swizzle.
bool encode_tma_2d_plain(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows,
                         uint32_t box_inner, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(ptr), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// Row-major [rows, K] 16-bit matrix, box = 64 K-elements x box_rows rows.
bool make_map_2d(CUtensorMap *m, int dtype, const void *ptr, uint64_t K, uint64_t rows,
                 uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {K * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Stacked [E, rows, K] 16-bit weights, box = 64 K-elements x box_rows rows x 1 expert.
bool make_map_3d(CUtensorMap *m, int dtype, const void *ptr, uint64_t K, uint64_t rows,
                 uint64_t E, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {K, rows, E};
    cuuint64_t strides[2] = {K * 2, rows * K * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int DT, int MODE>
cudaError_t launch_typed(const CUtensorMap *maps, const GemmParams &p, int grid, cudaStream_t stream) {
    auto kern = grouped_gemm_kernel<DT, MODE>;
    // the shared-memory opt-in is set once per device (cheap launches, and no
    // attribute call while a graph is being captured after the first use)
    static std::atomic<bool> attr_done[64];  // zero-initialised; several host threads may launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<MODE>::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    return launch_pdl(kern, dim3(grid), dim3(NUM_THREADS), Layout<MODE>::SMEM, stream, maps[0], maps[1],
                      maps[2], maps[3], maps[4], maps[5], p);
}

template <int MODE>
cudaError_t launch_mode(int dtype, const CUtensorMap *maps, const GemmParams &p, int64_t tiles,
                        cudaStream_t stream) {
    const int grid = Layout<MODE>::MLP ? mlp_grid(tiles)
                                       : static_cast<int>(tiles < device_sm_count() ? tiles : device_sm_count());
    if (dtype == kBF16) return launch_typed<kBF16, MODE>(maps, p, grid, stream);
    return launch_typed<kF16, MODE>(maps, p, grid, stream);
}

GemmParams base_params(const int32_t *sizes, const int32_t *offsets, const int32_t *padded,
                       const int32_t *gidx, int64_t m_blocks, const float *row_weights, int32_t *err) {
    GemmParams p{};
    p.sizes = sizes;
    p.offsets = offsets;
    p.padded = padded;
    p.gidx = gidx;
    p.row_weights = row_weights;
    p.ready = nullptr;
    p.tile_counter = nullptr;
    p.gather_idx = nullptr;
    p.m_blocks = static_cast<int>(m_blocks);
    p.err = err;
    return p;
}

PhaseParams phase_params(void *out, int64_t K, int64_t N, int out_n) {
    PhaseParams ph;
    ph.out = out;
    ph.n_tiles = static_cast<int>((N + out_n - 1) / out_n);
    ph.k_blocks = static_cast<int>((K + BK - 1) / BK);
    ph.N = static_cast<int>(N);
    return ph;
}

// Stage-1 maps into maps[0..2]: rows [n_rows, d_h], W_gate / W_up [E, d_e, d_h].
bool stage1_maps(CUtensorMap *maps, int dtype, const void *a, const void *w_gate, const void *w_up,
                 int64_t n_rows, int64_t d_h, int64_t d_e, int64_t E) {
    return make_map_2d(&maps[0], dtype, a, static_cast<uint64_t>(d_h), static_cast<uint64_t>(n_rows), BM) &&
           make_map_3d(&maps[1], dtype, w_gate, static_cast<uint64_t>(d_h), static_cast<uint64_t>(d_e),
                       static_cast<uint64_t>(E), 128u) &&
           make_map_3d(&maps[2], dtype, w_up, static_cast<uint64_t>(d_h), static_cast<uint64_t>(d_e),
                       static_cast<uint64_t>(E), 128u);
}

// Stage-2 maps into maps[3..4]: h [n_rows, d_e] (boxes of h_rows rows),
// W_down [E, d_h, d_e].
bool stage2_maps(CUtensorMap *maps, int dtype, const void *h, const void *w_down, int64_t n_rows,
                 int64_t d_h, int64_t d_e, int64_t E, uint32_t h_rows = BM) {
    return make_map_2d(&maps[3], dtype, h, static_cast<uint64_t>(d_e), static_cast<uint64_t>(n_rows), h_rows) &&
           make_map_3d(&maps[4], dtype, w_down, static_cast<uint64_t>(d_e), static_cast<uint64_t>(d_h),
                       static_cast<uint64_t>(E), 256u);
}

}  // namespace

cudaError_t launch_grouped_gemm(bool gate_up, int dtype, const void *a, const void *w0,
                                const void *w1, const int32_t *sizes, const int32_t *offsets,
                                const int32_t *padded, const int32_t *gidx, int64_t m_blocks,
                                const float *row_weights, int64_t n_rows, int64_t K, int64_t N,
                                int64_t E, void *out, int32_t *err, cudaStream_t stream) {
    if (n_rows <= 0 || m_blocks <= 0) return cudaSuccess;
    CUtensorMap maps[6];
    GemmParams p = base_params(sizes, offsets, padded, gidx, m_blocks, row_weights, err);
    if (gate_up) {
        // stage 1: K = d_h, N = d_e
        if (!stage1_maps(maps, dtype, a, w0, w1, n_rows, K, N, E)) return cudaErrorInvalidValue;
        maps[3] = maps[0];
        maps[4] = maps[1];
        maps[5] = maps[0];
        p.ph[0] = phase_params(out, K, N, 128);
        p.ph[1] = p.ph[0];
        return launch_mode<MODE_GATE_UP>(dtype, maps, p, m_blocks * p.ph[0].n_tiles, stream);
    }
    // stage 2: K = d_e, N = d_h
    if (!stage2_maps(maps, dtype, a, w0, n_rows, N, K, E)) return cudaErrorInvalidValue;
    maps[0] = maps[3];
    maps[1] = maps[4];
    maps[2] = maps[4];
    maps[5] = maps[3];
    p.ph[1] = phase_params(out, K, N, 256);
    p.ph[0] = p.ph[1];
    return launch_mode<MODE_DOWN>(dtype, maps, p, m_blocks * p.ph[1].n_tiles, stream);
}

cudaError_t launch_grouped_mlp(int dtype, const void *a, const void *w_gate, const void *w_up,
                               const void *w_down, const int32_t *sizes, const int32_t *offsets,
                               const int32_t *padded, const int32_t *gidx, int64_t m_blocks,
                               const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                               int64_t E, void *h, void *y, int32_t *ready, int32_t *err,
                               cudaStream_t stream, const void *x, const int32_t *gather_idx,
                               int64_t T) {
    if (n_rows <= 0 || m_blocks <= 0) return cudaSuccess;
    // rows gathered from at most 64 tokens: no expert, so no block, holds
    // more than 64 rows (MODE_MLP_FEW; its stage 2 copies 64 rows of h)
    const bool few = gather_idx != nullptr && T <= SWAP_MAX_ROWS;
    CUtensorMap maps[6];
    // gathering: stage 1 reads token rows of x by index (then `a` is unused)
    const void *a_map = gather_idx ? x : a;
    const int64_t a_rows = gather_idx ? T : n_rows;
    if (!stage1_maps(maps, dtype, a_map, w_gate, w_up, a_rows, d_h, d_e, E) ||
        !stage2_maps(maps, dtype, h, w_down, n_rows, d_h, d_e, E, few ? SWAP_MAX_ROWS : BM))
        return cudaErrorInvalidValue;
    if (gather_idx) {
        if (!make_map_2d(&maps[5], dtype, x, static_cast<uint64_t>(d_h), static_cast<uint64_t>(T), 1u))
            return cudaErrorInvalidValue;
    } else {
        maps[5] = maps[0];
    }
    GemmParams p = base_params(sizes, offsets, padded, gidx, m_blocks, row_weights, err);
    p.ready = ready;
    p.tile_counter = ready + m_blocks;
    p.gather_idx = gather_idx;
    p.prefetch_experts = few ? static_cast<int>(E) : 0;
    p.ph[0] = phase_params(h, d_h, d_e, 128);
    p.ph[1] = phase_params(y, d_e, d_h, 256);
    const int64_t tiles = m_blocks * (p.ph[0].n_tiles + p.ph[1].n_tiles);
    if (few) return launch_mode<MODE_MLP_FEW>(dtype, maps, p, tiles, stream);
    return launch_mode<MODE_MLP>(dtype, maps, p, tiles, stream);
}

}  // namespace moe

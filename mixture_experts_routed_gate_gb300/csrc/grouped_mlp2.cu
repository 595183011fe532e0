// grouped_mlp2.cu -- both expert GEMM stages of the routed MoE forward in one
// persistent launch on CTA pairs: every tile is computed by two SMs with
// tcgen05.mma.cta_group::2 (M = 256), for many-token (prefill) problems.
//
// Stage 1 (CSDN "tilelang kernel stage 1 gate+up"):
//   h[rows of an expert] = silu(A W_gate[g]^T) * (A W_up[g]^T)
// Stage 2 (CSDN "tilelang kernel stage 2 down"):
//   y[rows of an expert] = h W_down[g]^T
// over the rows the dispatch tables assign to each expert.  Results equal the
// one-SM expert MLP of grouped_gemm.cu (each output element is one fp32 sum
// over K in the same tensor-core order, rounded once).
//
// Why pairs: a one-SM tile of 128 rows x 256 weight rows moves 48 KB of
// operands per 64-wide K step through one SM; split over two SMs, each SM
// moves 32 KB for the same multiply-adds (its 128 rows and half of the
// weight rows), so a 227 KB shared memory holds six steps in flight instead
// of four, and the tensor pipe waits less on operands.
//
// Work units, from the dispatch tables:
//   * big unit: 256 consecutive rows of an expert with more than 64 rows
//     (its last unit ragged).  Stage-1 tiles: 128 output features; CTA r
//     loads its 128 rows and W_gate (r = 0) or W_up (r = 1) rows of those
//     features, so each CTA's accumulator holds gate | up for its rows.
//     Stage-2 tiles: 256 output features; CTA r loads its 128 rows of h and
//     W_down rows [n0 + 128 r, +128).
//   * small unit: the rows (at most 64) of an expert with at most 64 rows,
//     computed swapped: the weights are the M = 256 operand, the rows the N
//     operand (rounded up to 16, half in each CTA).  Stage-1 tiles: 256
//     features, CTA r holding W_gate and W_up rows [n0 + 128 r, +128) (two
//     MMAs per K step: gate and up into two column ranges); stage-2 tiles:
//     512 features, CTA r holding W_down rows [n0 + 128 r, +128) and
//     [n0 + 256 + 128 r, +128).
// Tile order: all stage-1 tiles, then all stage-2 tiles; inside a stage the
// big units' tiles (expert by expert, weight stripe major: every unit of an
// expert on stripe n before stripe n + 1) interleaved evenly with the small
// units' tiles.  The even CTA of a pair takes tiles from a shared counter, in
// order, and hands each id to both CTAs; a stage-2 tile waits until every
// stage-1 epilogue warp of its unit has stored its h (per-unit counters), and
// since tiles are taken in order, those stage-1 tiles belong to running pairs.
//
// Roles per CTA (224 threads): warp 0 TMA producer (both CTAs load their own
// halves; the copies complete on the even CTA's ring barrier), warps 1 and 6
// MMA issuers (even CTA only: one thread each; they commit to both CTAs'
// barriers), warps 2-5 epilogue (each CTA drains its own tensor memory:
// SiLU(gate) * up or the down output, rounded to the dtype, stores of valid
// rows only).  One thread issues a small-N MMA about every 85 cycles, and a
// swapped tile needs one MMA per 4 KB of weights per SM, so a swapped tile's
// two accumulators (gate and up, or the two W_down halves) are issued by two
// threads in parallel, each in the same K order as one thread would (the
// results do not change); a big tile's MMAs (N = 256, bound by the tensor
// pipe) all come from warp 1, warp 6 only keeping step.  Every wait is
// bounded (2 s): on expiry the kernel records a timeout, winds down and
// returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int P_BK = 64;
constexpr int P_ST = 6;                     // ring stages
constexpr int P_R0 = 128 * P_BK * 2;        // 16 KB: rows (big) or weights (small)
constexpr int P_R1 = 128 * P_BK * 2;        // 16 KB: weights
constexpr int P_RT = 32;                    // token rows of a small tile per CTA
constexpr int P_R2 = P_RT * P_BK * 2;       // 4 KB: rows (small)
constexpr int P_STAGE = P_R0 + P_R1 + P_R2;  // 36 KB
constexpr int P_THREADS = 224;               // 7 warps (see the roles below)
constexpr int P_MMA2_WARP = 6;              // the second MMA issuer
constexpr int P_EPI = 4;
constexpr int P_TRING = 4;
constexpr int P_NEXT_FETCH = 2;
constexpr int P_MAX_UNITS = 512;
constexpr int P_SMALL_MAX = 64;
constexpr int P_BAR_BYTES = 256;
constexpr int P_SCHED_BYTES = P_MAX_UNITS * (4 + 4 + 4 + 2 + 2 + 2) + 64;
constexpr int P_SMEM = 1024 + P_ST * P_STAGE + P_BAR_BYTES + P_SCHED_BYTES;
static_assert(P_SMEM <= 227 * 1024, "shared memory per CTA");
static_assert(P_STAGE % 1024 == 0 && P_R0 % 1024 == 0 && (P_R0 + P_R1) % 1024 == 0, "swizzle atoms");

struct Mlp2Params {
    const int32_t *sizes;
    const int32_t *offsets;
    const int32_t *padded;
    int *ready;         // per unit (indexed by its first M block + window): stage-1 warp-tiles stored
    int *tile_counter;  // next tile to take
    void *h;            // [n_rows, d_e]
    void *y;            // [n_rows, d_h]
    int E, d_h, d_e;
    int kb1, kb2;                 // 64-wide K steps of stage 1 (d_h) and stage 2 (d_e)
    int nt1_big, nt1_small;       // stage-1 tiles per unit: d_e / 128, d_e / 256
    int nt2_big, nt2_small;       // stage-2 tiles per unit: d_h / 256, d_h / 512
    int *err;
};

struct Unit {
    int g, m_start, rows, ctr;
};

struct Sched {
    const int *g, *m, *ctr;
    const uint16_t *rows;
    const int16_t *run_start, *run_len;
    int n_big, n_small;
};

struct PTile {
    int phase;  // 0 gate/up, 1 down
    bool big;
    int unit, n0;
    Unit u;
};

__device__ __forceinline__ PTile decode_ptile(const Mlp2Params &p, const Sched &sc, int tile) {
    const int64_t bt1 = static_cast<int64_t>(sc.n_big) * p.nt1_big, st1 = static_cast<int64_t>(sc.n_small) * p.nt1_small;
    PTile t;
    int64_t i = tile;
    t.phase = 0;
    if (i >= bt1 + st1) {
        t.phase = 1;
        i -= bt1 + st1;
    }
    const int ntb = t.phase ? p.nt2_big : p.nt1_big;
    const int nts = t.phase ? p.nt2_small : p.nt1_small;
    const int64_t bt = static_cast<int64_t>(sc.n_big) * ntb, st = static_cast<int64_t>(sc.n_small) * nts;
    const int64_t all = bt + st;
    const int64_t hb = i * bt / all, hn = (i + 1) * bt / all;  // big tiles before position i
    if (hn > hb) {
        t.big = true;
        const int fb = static_cast<int>(hb / ntb);  // a big unit of the run holding big tile hb
        const int rs = sc.run_start[fb], rl = sc.run_len[fb];
        const int64_t o = hb - static_cast<int64_t>(rs) * ntb;
        const int nt = static_cast<int>(o / rl);
        t.unit = rs + static_cast<int>(o - static_cast<int64_t>(nt) * rl);
        t.n0 = nt * (t.phase ? 256 : 128);
    } else {
        t.big = false;
        const int64_t l = i - hb;
        t.unit = sc.n_big + static_cast<int>(l / nts);
        t.n0 = static_cast<int>(l % nts) * (t.phase ? 512 : 256);
    }
    t.u.g = sc.g[t.unit];
    t.u.m_start = sc.m[t.unit];
    t.u.rows = sc.rows[t.unit];
    t.u.ctr = sc.ctr[t.unit];
    return t;
}

// Exclusive scan of one int per thread across the CTA; returns the total.
__device__ __forceinline__ int p_scan(int v, int *scratch, int *total) {
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
    for (int w = 0; w < P_THREADS / 32; ++w) {
        const int x = scratch[w];
        if (w < warp) base += x;
        tot += x;
    }
    __syncthreads();
    *total = tot;
    return base + incl - v;
}

__device__ __forceinline__ void p_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long start = global_timer_ns();
    while (!mbar_try_wait_cluster(bar, parity))
        if (global_timer_ns() - start > kWaitTimeoutNs) return;
}

template <int DT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    grouped_mlp2_kernel(const __grid_constant__ CUtensorMap tmA,   // rows [n_rows, d_h], box 64 x 128
                        const __grid_constant__ CUtensorMap tmAs,  // rows, box 64 x 32
                        const __grid_constant__ CUtensorMap tmWg,  // W_gate [E, d_e, d_h], box 64 x 128
                        const __grid_constant__ CUtensorMap tmWu,  // W_up, same
                        const __grid_constant__ CUtensorMap tmH,   // h [n_rows, d_e], box 64 x 128
                        const __grid_constant__ CUtensorMap tmHs,  // h, box 64 x 32
                        const __grid_constant__ CUtensorMap tmWd,  // W_down [E, d_h, d_e], box 64 x 128
                        const Mlp2Params p) {
    constexpr uint32_t IDESC_BIG = idesc_f16(DT == kBF16, 256, 256);
    using OutT = typename Elem<DT>::T;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + P_ST * P_STAGE);
    constexpr int NBARS = 2 * P_ST + 4 + 2 * P_TRING;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *tid_ring = reinterpret_cast<int *>(tmem_slot + 2);
    static_assert(NBARS * 8 + 8 + 4 * P_TRING <= P_BAR_BYTES, "barrier area");
    int *u_g = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + P_BAR_BYTES);
    int *u_m = u_g + P_MAX_UNITS;
    int *u_ctr = u_m + P_MAX_UNITS;
    uint16_t *u_rows = reinterpret_cast<uint16_t *>(u_ctr + P_MAX_UNITS);
    int16_t *u_rs = reinterpret_cast<int16_t *>(u_rows + P_MAX_UNITS);
    int16_t *u_rl = u_rs + P_MAX_UNITS;
    int *scan_scratch = reinterpret_cast<int *>(u_rl + P_MAX_UNITS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();
    const bool leader = rank == 0;
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (P_ST + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * P_ST + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * P_ST + 2 + a); };
    auto tidf_bar = [&](int i) { return bar0 + 8u * (2 * P_ST + 4 + i); };
    auto tide_bar = [&](int i) { return bar0 + 8u * (2 * P_ST + 4 + P_TRING + i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_ST; ++s) {
            mbar_init(full_bar(s), 1);   // even CTA: its expect_tx arrival (+ both CTAs' bytes)
            mbar_init(empty_bar(s), 2);  // the commits of the pair's two MMA threads
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 2);            // the commits of the two MMA threads
            mbar_init(tempty_bar(a), 2 * P_EPI);   // even CTA: every epilogue warp of both CTAs
        }
        for (int i = 0; i < P_TRING; ++i) {
            mbar_init(tidf_bar(i), 1);  // the even CTA's producer
            // even CTA: its two MMA threads and epilogue warps, the odd CTA's
            // producer and epilogue warps
            mbar_init(tide_bar(i), 3 + 2 * P_EPI);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmAs);
        tma_prefetch_desc(&tmWg);
        tma_prefetch_desc(&tmWu);
        tma_prefetch_desc(&tmH);
        tma_prefetch_desc(&tmHs);
        tma_prefetch_desc(&tmWd);
    }
    if (warp == 1) {
        tmem_alloc2(smem_u32(tmem_slot), 512);
        tmem_relinquish2();
    }
    griddep_wait();  // the tables, rows and counters come from earlier kernels
    griddep_launch_dependents();
    int first_tile = 0;
    if (leader && threadIdx.x == 0) first_tile = atomicAdd(p.tile_counter, 1);

    // ----- schedule: units from the tables (both CTAs build the same list) -----
    int n_big, n_small;
    {
        const int chunk = (p.E + P_THREADS - 1) / P_THREADS;
        const int lo = threadIdx.x * chunk, hi = min(p.E, lo + chunk);
        int nb = 0, ns = 0;
        for (int g = lo; g < hi; ++g) {
            const int sz = __ldg(p.sizes + g);
            if (sz > P_SMALL_MAX) nb += (sz + 255) / 256;
            else if (sz > 0) ns += 1;
        }
        int bb = p_scan(nb, scan_scratch, &n_big);
        int bs = p_scan(ns, scan_scratch, &n_small);
        if (n_big + n_small <= P_MAX_UNITS) {
            for (int g = lo; g < hi; ++g) {
                const int sz = __ldg(p.sizes + g);
                const int off = __ldg(p.offsets + g);
                const int blk = __ldg(p.padded + g) / 128;
                if (sz > P_SMALL_MAX) {
                    const int nw = (sz + 255) / 256;
                    for (int w = 0; w < nw; ++w) {
                        const int u = bb + w;
                        u_g[u] = g;
                        u_m[u] = off + 256 * w;
                        u_rows[u] = static_cast<uint16_t>(min(256, sz - 256 * w));
                        u_ctr[u] = blk + w;
                        u_rs[u] = static_cast<int16_t>(bb);
                        u_rl[u] = static_cast<int16_t>(nw);
                    }
                    bb += nw;
                } else if (sz > 0) {
                    const int u = n_big + bs++;
                    u_g[u] = g;
                    u_m[u] = off;
                    u_rows[u] = static_cast<uint16_t>(sz);
                    u_ctr[u] = blk;
                }
            }
        }
    }
    const bool sched_ok = n_big + n_small <= P_MAX_UNITS;
    if (!sched_ok && threadIdx.x == 0) {
        atomicExch(p.err, kErrDeviceFlag);  // the host admits no such problem
        *abort_flag = 1;
    }
    const Sched sc{u_g, u_m, u_ctr, u_rows, u_rs, u_rl, n_big, n_small};
    const int total = sched_ok ? static_cast<int>(static_cast<int64_t>(n_big) * (p.nt1_big + p.nt2_big) +
                                                  static_cast<int64_t>(n_small) * (p.nt1_small + p.nt2_small))
                               : 0;
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t peer = rank ^ 1u;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        const uint64_t pol_first = l2_policy_evict_first();
        const uint64_t pol_last = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        long issued = 0;
        bool ok = true;
        int rslot = 0;
        uint32_t rphase = 0;
        int next_tile = first_tile;
        bool have_next = true;
        for (;;) {
            // tile id: the even CTA takes it and writes it into both CTAs' rings
            int tile = -1, go = 1;
            if (lane == 0) {
                if (leader) {
                    if (!have_next) next_tile = atomicAdd(p.tile_counter, 1);
                    tile = next_tile;
                    have_next = false;
                    if (tile >= total) tile = -1;
                    go = mbar_wait_cluster_bounded(tide_bar(rslot), rphase ^ 1u, abort_flag, p.err) ? 1 : 0;
                    if (go) {
                        tid_ring[rslot] = tile;
                        st_shared_remote_u32(smem_map_rank(smem_u32(tid_ring + rslot), peer),
                                             static_cast<uint32_t>(tile));
                        mbar_arrive(tidf_bar(rslot));
                        mbar_arrive_remote(smem_map_rank(tidf_bar(rslot), peer));
                    }
                } else {
                    go = mbar_wait_cluster_bounded(tidf_bar(rslot), rphase, abort_flag, p.err) ? 1 : 0;
                    if (go) {
                        tile = tid_ring[rslot];
                        mbar_arrive_remote(smem_map_rank(tide_bar(rslot), 0));
                    }
                }
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (++rslot == P_TRING) {
                rslot = 0;
                rphase ^= 1u;
            }
            if (!go) {
                ok = false;
                break;
            }
            if (tile < 0) break;
            const PTile t = decode_ptile(p, sc, tile);
            if (t.phase == 1) {
                // this tile reads h rows of its unit: every stage-1 warp-tile stored
                const int target = 2 * P_EPI * (t.big ? p.nt1_big : p.nt1_small);
                if (lane == 0) go = counter_wait_bounded(p.ready + t.u.ctr, target, abort_flag, p.err) ? 1 : 0;
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
            }
            const int kblocks = t.phase ? p.kb2 : p.kb1;
            const int fetch_kb = kblocks > P_NEXT_FETCH ? kblocks - P_NEXT_FETCH : 0;
            const uint32_t bytes = static_cast<uint32_t>(2 * (t.big ? P_R0 + P_R1 : P_STAGE));
            const int half = ((t.u.rows + 15) & ~15) / 2;
            if (lane == 0) {
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (leader && kb == fetch_kb) {
                        next_tile = atomicAdd(p.tile_counter, 1);
                        have_next = true;
                    }
                    if (!mbar_wait_cluster_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full_bar(stage), bytes);
                    const uint32_t fb = smem_map_rank(full_bar(stage), 0);
                    const uint32_t r0 = smem_u32(ring + stage * P_STAGE);
                    const uint32_t r1 = r0 + P_R0, r2 = r1 + P_R1;
                    const int k0 = kb * P_BK;
                    if (t.big) {
                        // a large expert's rows and weight stripes are reused by its other tiles
                        if (t.phase == 0) {
                            tma2_load_2d_hint(r0, &tmA, fb, k0, t.u.m_start + 128 * static_cast<int>(rank), pol_last);
                            tma2_load_3d_hint(r1, rank ? &tmWu : &tmWg, fb, k0, t.n0, t.u.g, pol_last);
                        } else {
                            tma2_load_2d_hint(r0, &tmH, fb, k0, t.u.m_start + 128 * static_cast<int>(rank), pol_last);
                            tma2_load_3d_hint(r1, &tmWd, fb, k0, t.n0 + 128 * static_cast<int>(rank), t.u.g,
                                              pol_last);
                        }
                    } else {
                        // a small expert's weights are read by this unit only: let them leave L2 first
                        const int m0 = t.u.m_start + half * static_cast<int>(rank);
                        const int f0 = t.n0 + 128 * static_cast<int>(rank);
                        if (t.phase == 0) {
                            tma2_load_3d_hint(r0, &tmWg, fb, k0, f0, t.u.g, pol_first);
                            tma2_load_3d_hint(r1, &tmWu, fb, k0, f0, t.u.g, pol_first);
                            tma2_load_2d_hint(r2, &tmAs, fb, k0, m0, pol_last);
                        } else {
                            tma2_load_3d_hint(r0, &tmWd, fb, k0, f0, t.u.g, pol_first);
                            tma2_load_3d_hint(r1, &tmWd, fb, k0, f0 + 256, t.u.g, pol_first);
                            tma2_load_2d_hint(r2, &tmHs, fb, k0, m0, pol_last);
                        }
                    }
                    ++issued;
                    if (++stage == P_ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
        }
        if (!ok && leader && lane == 0) {
            // let the copies still in flight (this CTA's and the peer's) land
            for (long j = 1; j <= P_ST && j <= issued; ++j) {
                const long i = issued - j;
                p_drain(full_bar(static_cast<int>(i % P_ST)), static_cast<uint32_t>((i / P_ST) & 1));
            }
        }
    } else if (warp == 1 || warp == P_MMA2_WARP) {
        // ------------------------------- MMA issuers --------------------------------
        // thread A (warp 1): every MMA of a big tile, the first accumulator of a
        // swapped tile; thread B (warp 6): the second accumulator of a swapped
        // tile.  Both wait for each stage and commit it, so every barrier phase
        // sees one commit from each.
        const bool mma_b = warp == P_MMA2_WARP;
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            uint32_t last_bar = 0, last_parity = 0;
            bool committed = false;
            int rslot = 0;
            uint32_t rphase = 0;
            for (;;) {
                if (!mbar_wait_bounded(tidf_bar(rslot), rphase, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const int tile = tid_ring[rslot];
                mbar_arrive(tide_bar(rslot));
                if (++rslot == P_TRING) {
                    rslot = 0;
                    rphase ^= 1u;
                }
                if (tile < 0) break;
                const PTile t = decode_ptile(p, sc, tile);
                const int kblocks = t.phase ? p.kb2 : p.kb1;
                const int acc = local & 1;
                const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
                if (!mbar_wait_cluster_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
                const int np = (t.u.rows + 15) & ~15;
                const uint32_t idesc_sw = idesc_f16(DT == kBF16, 256, static_cast<uint32_t>(np));
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_cluster_bounded(full_bar(stage), phase, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t r0 = smem_u32(ring + stage * P_STAGE);
                    const uint64_t d0 = smem_desc_sw128(r0), d1 = smem_desc_sw128(r0 + P_R0),
                                   d2 = smem_desc_sw128(r0 + P_R0 + P_R1);
                    if (t.big) {
                        if (!mma_b) {
#pragma unroll
                            for (int k = 0; k < P_BK / 16; ++k)
                                tc_mma2_f16(d_tmem, d0 + 2u * k, d1 + 2u * k, IDESC_BIG, (kb | k) != 0 ? 1u : 0u);
                        }
                    } else {
                        // D[feature][row]: the R0 weights into columns [0, np) (thread A),
                        // R1 into [np, 2 np) (thread B)
                        const uint32_t d_acc = mma_b ? d_tmem + static_cast<uint32_t>(np) : d_tmem;
                        const uint64_t da = mma_b ? d1 : d0;
#pragma unroll
                        for (int k = 0; k < P_BK / 16; ++k)
                            tc_mma2_f16(d_acc, da + 2u * k, d2 + 2u * k, idesc_sw, (kb | k) != 0 ? 1u : 0u);
                    }
                    tc_commit2_both(empty_bar(stage));  // frees the stage in both CTAs
                    last_bar = empty_bar(stage);
                    last_parity = phase;
                    committed = true;
                    if (++stage == P_ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit2_both(tfull_bar(acc));  // both CTAs' accumulators ready
                ++local;
            }
            if (!ok && committed) p_drain(last_bar, last_parity);
        }
    } else {
        // --------------------------------- epilogue ---------------------------------
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        const int row = q * 32 + lane;
        const uint32_t tempty_leader = smem_map_rank(tempty_bar(0), 0);  // + 8 * acc
        int local = 0;
        int rslot = 0;
        uint32_t rphase = 0;
        for (;;) {
            int got = 1, tile = -1;
            if (lane == 0) {
                got = mbar_wait_cluster_bounded(tidf_bar(rslot), rphase, abort_flag, p.err) ? 1 : 0;
                if (got) {
                    tile = tid_ring[rslot];
                    if (leader) mbar_arrive(tide_bar(rslot));
                    else mbar_arrive_remote(smem_map_rank(tide_bar(rslot), 0));
                }
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (++rslot == P_TRING) {
                rslot = 0;
                rphase ^= 1u;
            }
            if (!got || tile < 0) break;
            const PTile t = decode_ptile(p, sc, tile);
            const bool gu = t.phase == 0;  // stage 1: silu(gate) * up
            const int N = gu ? p.d_e : p.d_h;
            OutT *const out_base = reinterpret_cast<OutT *>(gu ? p.h : p.y);
            const int acc = local & 1;
            const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
            int ready = 1;
            if (lane == 0) ready = mbar_wait_cluster_bounded(tfull_bar(acc), acc_phase, abort_flag, p.err) ? 1 : 0;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * 256);
            if (!t.big) {
                // swapped: this thread holds output feature f0 (and, for stage 2, f1)
                // for every row j of the unit
                const int np = (t.u.rows + 15) & ~15;
                const int f0 = t.n0 + 128 * static_cast<int>(rank) + row;
                const int f1 = gu ? -1 : f0 + 256;
#pragma unroll 1
                for (int j0 = 0; j0 < np; j0 += 16) {
                    uint32_t a[16], b[16];
                    tmem_ld16(t_row + j0, a);
                    tmem_ld16(t_row + np + j0, b);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        if (j < t.u.rows) {
                            const int64_t r = static_cast<int64_t>(t.u.m_start + j) * N;
                            if (gu) {
                                const float gv = __uint_as_float(a[jj]);
                                const float s = gv * __frcp_rn(1.0f + __expf(-gv));
                                if (f0 < N) out_base[r + f0] = from_f32<OutT>(s * __uint_as_float(b[jj]));
                            } else {
                                if (f0 < N) out_base[r + f0] = from_f32<OutT>(__uint_as_float(a[jj]));
                                if (f1 < N) out_base[r + f1] = from_f32<OutT>(__uint_as_float(b[jj]));
                            }
                        }
                    }
                }
            } else {
                const int li = 128 * static_cast<int>(rank) + row;  // row of the unit
                const bool valid = li < t.u.rows;
                OutT *out_row = out_base + static_cast<int64_t>(t.u.m_start + (valid ? li : 0)) * N;
                const int out_cols = gu ? 128 : 256;
#pragma unroll 1
                for (int c = 0; c < out_cols / 16; ++c) {
                    const int col = t.n0 + c * 16;
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
                            for (int hh = 0; hh < 2; ++hh) {
                                const float gv = __uint_as_float(g[2 * i + hh]);
                                const float uv = __uint_as_float(u[2 * i + hh]);
                                const float s = gv * __frcp_rn(1.0f + __expf(-gv));
                                v[hh] = s * uv;
                            }
                            packed[i] = pack2<DT>(v[0], v[1]);
                        }
                    } else {
                        uint32_t r[16];
                        tmem_ld16(t_row + c * 16, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            packed[i] = pack2<DT>(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    }
                    if (valid && col < N) {
                        uint4 *dst = reinterpret_cast<uint4 *>(out_row + col);
                        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(tempty_bar(acc));
                else mbar_arrive_remote(tempty_leader + 8u * static_cast<uint32_t>(acc));
            }
            if (gu) {
                // h stored: visible at gpu scope and to the async proxy, then counted
                __threadfence();
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) counter_publish(p.ready + t.u.ctr);
            }
            ++local;
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the pair's MMAs or arrivals may touch it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem_base, 512);
    }
}

template <int DT>
cudaError_t launch_mlp2_typed(const CUtensorMap *maps, const Mlp2Params &p, int grid, cudaStream_t stream) {
    auto kern = grouped_mlp2_kernel<DT>;
    static std::atomic<bool> attr_done[64];  // zero-initialised; several host threads may launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    return launch_pdl(kern, dim3(grid), dim3(P_THREADS), P_SMEM, stream, maps[0], maps[1], maps[2], maps[3],
                      maps[4], maps[5], maps[6], p);
}

bool map2d(CUtensorMap *m, int dtype, const void *ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    const int dt = dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t dims[2] = {inner, rows};
    const uint64_t strides[1] = {inner * 2};
    const uint32_t box[2] = {P_BK, box_rows};
    return encode_tma_map(m, dt, 2, ptr, dims, strides, box, 1);
}

bool map3d(CUtensorMap *m, int dtype, const void *ptr, uint64_t inner, uint64_t rows, uint64_t E) {
    const int dt = dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t dims[3] = {inner, rows, E};
    const uint64_t strides[2] = {inner * 2, rows * inner * 2};
    const uint32_t box[3] = {P_BK, 128, 1};
    return encode_tma_map(m, dt, 3, ptr, dims, strides, box, 1);
}

}  // namespace

bool grouped_mlp2_applies(int64_t n_rows, int64_t d_h, int64_t d_e, int64_t E) {
    // units: at most n_rows / 256 + E (a ragged window per big expert)
    return device_sm_count() >= 2 && d_e % 256 == 0 && d_h % 512 == 0 && n_rows / 256 + E <= P_MAX_UNITS;
}

cudaError_t launch_grouped_mlp2(int dtype, const void *a, const void *w_gate, const void *w_up,
                                const void *w_down, const int32_t *sizes, const int32_t *offsets,
                                const int32_t *padded, int64_t m_blocks, int64_t n_rows, int64_t d_h,
                                int64_t d_e, int64_t E, void *h, void *y, int32_t *ready, int32_t *err,
                                cudaStream_t stream) {
    if (n_rows <= 0 || m_blocks <= 0) return cudaSuccess;
    CUtensorMap maps[7];
    const uint64_t R = static_cast<uint64_t>(n_rows), H = static_cast<uint64_t>(d_h), D = static_cast<uint64_t>(d_e),
                   NE = static_cast<uint64_t>(E);
    if (!map2d(&maps[0], dtype, a, H, R, 128) || !map2d(&maps[1], dtype, a, H, R, P_RT) ||
        !map3d(&maps[2], dtype, w_gate, H, D, NE) || !map3d(&maps[3], dtype, w_up, H, D, NE) ||
        !map2d(&maps[4], dtype, h, D, R, 128) || !map2d(&maps[5], dtype, h, D, R, P_RT) ||
        !map3d(&maps[6], dtype, w_down, D, H, NE))
        return cudaErrorInvalidValue;
    Mlp2Params p{};
    p.sizes = sizes;
    p.offsets = offsets;
    p.padded = padded;
    p.ready = ready;
    p.tile_counter = ready + m_blocks;
    p.h = h;
    p.y = y;
    p.E = static_cast<int>(E);
    p.d_h = static_cast<int>(d_h);
    p.d_e = static_cast<int>(d_e);
    p.kb1 = static_cast<int>(d_h / P_BK);
    p.kb2 = static_cast<int>(d_e / P_BK);
    p.nt1_big = static_cast<int>(d_e / 128);
    p.nt1_small = static_cast<int>(d_e / 256);
    p.nt2_big = static_cast<int>(d_h / 256);
    p.nt2_small = static_cast<int>(d_h / 512);
    p.err = err;
    // pairs of CTAs, one CTA per SM; MOE_MLP_GRID (tests) may ask for another count
    int grid = mlp_grid(int64_t(1) << 30);
    grid = grid < 2 ? 2 : grid & ~1;
    if (dtype == kBF16) return launch_mlp2_typed<kBF16>(maps, p, grid, stream);
    return launch_mlp2_typed<kF16>(maps, p, grid, stream);
}

}  // namespace moe

/*
 * moe_oracle.c -- plain, slow, obviously-correct CPU oracle of the routed-expert
 * MoE forward (gate -> top-k -> dispatch tables -> grouped gate/up + SiLU ->
 * grouped down -> moe_reduce_fused combine).
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check of the entry module and
 * the CPU-baseline / reference legs of the benchmark load this library.  It
 * shares no code, header, table or helper with the CUDA library; neither side
 * includes or links the other.
 *
 * Sources.  Each function names the passage it follows:
 *   [CSDN]  "tilelang baseline" article on the tilelang-metax MoE contest
 *           operator (devpress.csdn.net): sections "MoE" (buffers), "forward"
 *           (routing, sort, tables, scatter-reduce), "tilelang kernel stage 1
 *           gate+up" and "tilelang kernel stage 2 down".
 *   [SKEL]  TileLang tutorial ch.18 skeletons.py, moe_routed_kernel (the
 *           dispatch contract and the two kernels), w4a8_dequant_gemm (the
 *           int4 weight format) and the module notes on quantisation.
 *   [PR55]  TileOPs-Metax PR #55 "[moe_reduce_fused] feat": section 1
 *           (kernel semantics), section 2 (accuracy), section 3 (roofline).
 *   The gate body is not printed on any page; its reading (softmax over fp32
 *   logits, top-k with ties to the lower expert id, the top-k probabilities as
 *   weights, and the lane/butterfly summation order of the logits) is stated at
 *   oracle_gate_logits and oracle_topk_softmax.
 *
 * Precision.  Where the pages fix it (fp32 accumulators of both GEMM stages and
 * of the combine; activations and intermediates stored in the activation
 * dtype) this file uses it, summing in plain ascending order.  Where they do
 * not (the softmax, the SiLU), it uses double and rounds once.
 *
 * Parity status: every function here is pinned by the CPU tests (worked
 * examples from the pages, brute force, closed forms, library routines).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_F16 0
#define OR_BF16 1
#define OR_F32 2
#define OR_E4M3 3

#define OR_OK 0
#define OR_EINVAL 1

/* ------------------------------------------------------------------------- */
/* IEEE-754 storage conversions, written from the binary16 / bfloat16 formats. */
/* ------------------------------------------------------------------------- */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.  Exact widening. */
static float half_to_float(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t exp = (uint32_t)(h >> 10) & 0x1fu;
    uint32_t frac = (uint32_t)h & 0x3ffu;
    double mag;
    if (exp == 0x1f) {
        if (frac == 0) return sign ? -INFINITY : INFINITY;
        return bits_f32((sign << 31) | 0x7fc00000u | (frac << 13));
    }
    if (exp == 0) mag = ldexp((double)frac, -24);                 /* subnormal */
    else mag = ldexp((double)(frac | 0x400u), (int)exp - 25);      /* normal    */
    return (float)(sign ? -mag : mag);                             /* exact     */
}

/* Round a finite binary32 value to binary16, round-to-nearest-even. */
static uint16_t float_to_half(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    double a = fabs((double)f);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    if (isinf(f)) return (uint16_t)(sign | 0x7c00u);
    /* Largest finite half is 65504; values >= 65520 round to infinity. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: units of 2^-24, ties to even */
        double q = a * ldexp(1.0, 24);
        double r = nearbyint(q); /* default rounding mode: nearest-even */
        return (uint16_t)(sign | (uint16_t)r);  /* r == 1024 gives the min normal */
    }
    int e;
    double m = frexp(a, &e);         /* a = m * 2^e, m in [0.5, 1) */
    /* significand with 11 bits: a = s * 2^(e-11), s in [1024, 2048) */
    double s = nearbyint(ldexp(m, 11));
    if (s >= 2048.0) { s = 1024.0; e += 1; }
    int biased = e - 1 + 15;
    if (biased >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)((uint32_t)s - 1024u));
}

/* bfloat16 is the top half of binary32.  Exact widening. */
static float bf16_to_float(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* Round binary32 to bfloat16, round-to-nearest-even; NaN stays quiet NaN. */
static uint16_t float_to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;  /* carry into the exponent gives inf correctly */
}

/* Every binary16 pattern widened once (the table is half_to_float itself). */
static float g_half_table[65536];
static pthread_once_t g_half_once = PTHREAD_ONCE_INIT;
static void fill_half_table(void)
{
    for (uint32_t b = 0; b < 65536u; ++b) g_half_table[b] = half_to_float((uint16_t)b);
}

/* float8 e4m3fn: 1 sign, 4 exponent (bias 7), 3 fraction bits; no infinity;
 * S.1111.111 is NaN; largest finite 448, smallest subnormal 2^-9. */
static float e4m3_to_float(uint8_t b)
{
    uint32_t sign = (b >> 7) & 1u, exp = (b >> 3) & 0xfu, frac = b & 7u;
    double mag;
    if (exp == 0xf && frac == 7) return bits_f32((sign << 31) | 0x7fc00000u);
    if (exp == 0) mag = ldexp((double)frac, -9);
    else mag = ldexp((double)(8u | frac), (int)exp - 10);
    return (float)(sign ? -mag : mag);
}

/* Round to e4m3fn, nearest-even, saturating finite values to +-448; NaN -> NaN. */
static uint8_t float_to_e4m3_sat(float f)
{
    uint8_t sign = (uint8_t)((f32_bits(f) >> 24) & 0x80u);
    if (isnan(f)) return (uint8_t)(sign | 0x7fu);
    double a = fabs((double)f);
    if (a >= 464.0) return (uint8_t)(sign | 0x7eu);     /* 448: rounds past the top */
    if (a < ldexp(1.0, -6)) {                            /* subnormal: units of 2^-9 */
        double r = nearbyint(a * ldexp(1.0, 9));
        return (uint8_t)(sign | (uint8_t)r);            /* r == 8 is the min normal */
    }
    int e;
    double m = frexp(a, &e);                             /* a = m * 2^e, m in [0.5, 1) */
    double sgn = nearbyint(ldexp(m, 4));                 /* 4 significant bits: [8, 16] */
    if (sgn >= 16.0) { sgn = 8.0; e += 1; }
    int biased = e + 6;
    return (uint8_t)(sign | (uint8_t)(biased << 3) | (uint8_t)((unsigned)sgn - 8u));
}

static float load_elem(const void *p, int64_t i, int dtype)
{
    if (dtype == OR_F16) return g_half_table[((const uint16_t *)p)[i]];
    if (dtype == OR_BF16) return bf16_to_float(((const uint16_t *)p)[i]);
    if (dtype == OR_E4M3) return e4m3_to_float(((const uint8_t *)p)[i]);
    return ((const float *)p)[i];
}

static void store_elem(void *p, int64_t i, int dtype, float v)
{
    if (dtype == OR_F16) ((uint16_t *)p)[i] = float_to_half(v);
    else if (dtype == OR_BF16) ((uint16_t *)p)[i] = float_to_bf16(v);
    else if (dtype == OR_E4M3) ((uint8_t *)p)[i] = float_to_e4m3_sat(v);
    else ((float *)p)[i] = v;
}

static int dtype_ok(int d) { return d == OR_F16 || d == OR_BF16 || d == OR_F32; }
static int out_dtype_ok(int d) { return dtype_ok(d) || d == OR_E4M3; }

static void oracle_init(void) { pthread_once(&g_half_once, fill_half_table); }

void oracle_decode(const void *src, int dtype, int64_t n, float *dst)
{
    oracle_init();
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, i, dtype);
}

void oracle_encode(const float *src, int dtype, int64_t n, void *dst)
{
    oracle_init();
    for (int64_t i = 0; i < n; ++i) store_elem(dst, i, dtype, src[i]);
}

/* ------------------------------------------------------------------------- */
/* A tiny fork/join helper: run fn(lo, hi, ctx) over [0, n) on nthreads.       */
/* ------------------------------------------------------------------------- */

typedef void (*range_fn)(int64_t lo, int64_t hi, void *ctx);
typedef struct { range_fn fn; void *ctx; int64_t lo, hi; } range_job;

static void *range_thread(void *arg)
{
    range_job *j = (range_job *)arg;
    j->fn(j->lo, j->hi, j->ctx);
    return NULL;
}

static int resolve_threads(int nthreads)
{
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void *ctx)
{
    int nt = resolve_threads(nthreads);
    if (nt > n) nt = (int)(n > 0 ? n : 1);
    if (nt <= 1) { fn(0, n, ctx); return; }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    range_job *jobs = (range_job *)malloc(sizeof(range_job) * (size_t)nt);
    int64_t per = (n + nt - 1) / nt;
    int started = 0;
    for (int t = 0; t < nt; ++t) {
        int64_t lo = (int64_t)t * per, hi = lo + per;
        if (hi > n) hi = n;
        if (lo >= hi) break;
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].lo = lo; jobs[t].hi = hi;
        if (pthread_create(&th[t], NULL, range_thread, &jobs[t]) != 0) {
            fn(lo, hi, ctx);          /* could not start a thread: run inline */
            jobs[t].fn = NULL;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; ++t)
        if (jobs[t].fn) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
}

int oracle_resolve_threads(int nthreads) { return resolve_threads(nthreads); }

/* ------------------------------------------------------------------------- */
/* o1: gate logits.                                                           */
/* ------------------------------------------------------------------------- */
/*
 * [CSDN "forward"]: expert_indices, expert_scores = gating_network(x); the
 * gate body is not printed.  Reading: a linear gate, logits l[t,e] =
 * sum_j x[t,j] * Wg[e,j] (+ bias[e]) in fp32.  The summation order is fixed
 * so that the routing decision is reproducible bit for bit:
 *   - the d_hidden axis is cut into chunks of 8 consecutive elements; chunk c
 *     belongs to lane (c mod 32);
 *   - each lane L sums its elements in ascending j: p_L = fmaf(x_j, w_j, p_L)
 *     starting from +0.0f;
 *   - the 32 partials are combined pairwise: for s = 16, 8, 4, 2, 1 every lane
 *     sets p_L = p_L + p_(L xor s) (all lanes updated from the old values);
 *   - the logit is p_0, plus bias[e] when a bias is given.
 * Requires d_hidden % 256 == 0.
 */
typedef struct {
    const void *x, *wg; const float *bias; int64_t d_h, E; int dtype; float *logits;
    const float *xf, *wf;
} gate_ctx;

static void gate_rows(int64_t lo, int64_t hi, void *vctx)
{
    gate_ctx *c = (gate_ctx *)vctx;
    const int64_t d_h = c->d_h;
    for (int64_t t = lo; t < hi; ++t) {
        const float *xr = c->xf + t * d_h;
        for (int64_t e = 0; e < c->E; ++e) {
            const float *wr = c->wf + e * d_h;
            float p[32];
            for (int L = 0; L < 32; ++L) p[L] = 0.0f;
            for (int64_t chunk = 0; chunk < d_h / 8; ++chunk) {
                int L = (int)(chunk % 32);
                for (int64_t j = chunk * 8; j < chunk * 8 + 8; ++j)
                    p[L] = fmaf(xr[j], wr[j], p[L]);
            }
            for (int s = 16; s >= 1; s >>= 1) {
                float q[32];
                for (int L = 0; L < 32; ++L) q[L] = p[L] + p[L ^ s];
                for (int L = 0; L < 32; ++L) p[L] = q[L];
            }
            float l = p[0];
            if (c->bias) l = l + c->bias[e];
            c->logits[t * c->E + e] = l;
        }
    }
}

int oracle_gate_logits(const void *x, const void *wg, const float *bias, int64_t T,
                       int64_t d_h, int64_t E, int dtype, float *logits, int nthreads)
{
    oracle_init();
    if (!x || !wg || !logits || T < 0 || E <= 0 || d_h <= 0 || d_h % 256 != 0 ||
        !dtype_ok(dtype))
        return OR_EINVAL;
    float *xf = (float *)malloc(sizeof(float) * (size_t)(T * d_h + 1));
    float *wf = (float *)malloc(sizeof(float) * (size_t)(E * d_h));
    if (!xf || !wf) { free(xf); free(wf); return OR_EINVAL; }
    oracle_decode(x, dtype, T * d_h, xf);
    oracle_decode(wg, dtype, E * d_h, wf);
    gate_ctx c = {x, wg, bias, d_h, E, dtype, logits, xf, wf};
    parallel_for(T, nthreads, gate_rows, &c);
    free(xf);
    free(wf);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* o2: top-k selection and softmax weights.                                   */
/* ------------------------------------------------------------------------- */
/*
 * [CSDN "forward"]: the gate returns expert_indices and expert_scores of shape
 * [B, S, top_k].  Reading: experts are ranked by (logit descending, expert id
 * ascending) and the first k are taken in that order; since softmax is
 * monotone this is the same ranking as by probability.  The weight of a
 * selected expert is its softmax probability over all E logits, with no
 * renormalisation over the k selected: w = exp(l - m) / sum_e exp(l_e - m),
 * m = max logit, computed in double and rounded once to fp32.
 */
static int ranks_before(float la, int64_t ia, float lb, int64_t ib)
{
    /* 1 when (la, ia) ranks strictly before (lb, ib) */
    return (la > lb) || (la == lb && ia < ib);
}

int oracle_topk_softmax(const float *logits, int64_t T, int64_t E, int64_t k,
                        int32_t *topk_idx, float *topk_w)
{
    if (!logits || !topk_idx || !topk_w || T < 0 || E <= 0 || k <= 0 || k > E)
        return OR_EINVAL;
    char *taken = (char *)malloc((size_t)E);
    if (!taken) return OR_EINVAL;
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        memset(taken, 0, (size_t)E);
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            topk_idx[t * k + j] = (int32_t)best;
        }
        double m = (double)l[topk_idx[t * k]];
        double denom = 0.0;
        for (int64_t e = 0; e < E; ++e) denom += exp((double)l[e] - m);
        for (int64_t j = 0; j < k; ++j)
            topk_w[t * k + j] = (float)(exp((double)l[topk_idx[t * k + j]] - m) / denom);
    }
    free(taken);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* o3: dispatch tables and the stable scatter.                                */
/* ------------------------------------------------------------------------- */

/* [CSDN "forward"] / [SKEL moe_routed_kernel]: M = ceil(B*S*top_k / block) + E */
int64_t oracle_num_m_blocks(int64_t T, int64_t k, int64_t E, int64_t block_m)
{
    if (T < 0 || k <= 0 || E <= 0 || block_m <= 0) return -1;
    return (T * k + block_m - 1) / block_m + E;
}

/*
 * [CSDN "forward"], steps 2-5:
 *   counts  = bincount(flat expert indices)            (reading: minlength = E)
 *   group_sizes[e]   = counts[e]
 *   group_offsets[e] = cumsum(counts)[e] - counts[e]   (exclusive prefix sum)
 *   group_padded_offsets[0] = 0,
 *   group_padded_offsets[i] = group_padded_offsets[i-1]
 *                             + ceil((counts[i-1] + 1) / block_m) * block_m
 *   group_idx_for_bx[bx] = the last i with bx*block_m >= group_padded_offsets[i]
 *                          (the double loop over bx and i, kept as written)
 * The sort "idxs = flat_expert_indices.argsort()" is read as a stable sort:
 * pair f = t*k + j goes to row r = group_offsets[e] + (number of pairs f' < f
 * with the same expert), sorted_token_idx[r] = f // k (the "idxs // top_k"
 * step), sorted_row_weight[r] = flat weight[f], token_topk_to_pos[f] = r.
 */
int oracle_build_dispatch(const int32_t *topk_idx, const float *topk_w, int64_t T,
                          int64_t k, int64_t E, int64_t block_m, int32_t *group_sizes,
                          int32_t *group_offsets, int32_t *group_padded_offsets,
                          int32_t *group_idx_for_bx, int64_t m_blocks,
                          int32_t *sorted_token_idx, float *sorted_row_weight,
                          int32_t *token_topk_to_pos)
{
    if (!topk_idx || !group_sizes || !group_offsets || !group_padded_offsets ||
        !group_idx_for_bx || T < 0 || k <= 0 || E <= 0 || block_m <= 0 ||
        m_blocks != oracle_num_m_blocks(T, k, E, block_m))
        return OR_EINVAL;
    const int64_t n_pairs = T * k;
    for (int64_t f = 0; f < n_pairs; ++f)
        if (topk_idx[f] < 0 || topk_idx[f] >= E) return OR_EINVAL;

    /* histogram (bincount with minlength E) */
    for (int64_t e = 0; e < E; ++e) group_sizes[e] = 0;
    for (int64_t f = 0; f < n_pairs; ++f) group_sizes[topk_idx[f]] += 1;

    /* inclusive cumsum, then offsets = cumsum - counts */
    int64_t running = 0;
    for (int64_t e = 0; e < E; ++e) {
        running += group_sizes[e];
        group_offsets[e] = (int32_t)(running - group_sizes[e]);
    }

    /* padded offsets */
    group_padded_offsets[0] = 0;
    for (int64_t i = 1; i < E; ++i) {
        int64_t c = group_sizes[i - 1];
        int64_t padded = ((c + 1 + block_m - 1) / block_m) * block_m;
        group_padded_offsets[i] = (int32_t)(group_padded_offsets[i - 1] + padded);
    }

    /* block -> expert lookup, as the double loop */
    for (int64_t bx = 0; bx < m_blocks; ++bx) {
        int64_t m_start_padded = bx * block_m;
        group_idx_for_bx[bx] = 0;
        for (int64_t i = 0; i < E; ++i)
            if (m_start_padded >= group_padded_offsets[i]) group_idx_for_bx[bx] = (int32_t)i;
    }

    /* stable scatter: walk the pairs in ascending f */
    if (sorted_token_idx || sorted_row_weight || token_topk_to_pos) {
        int64_t *next = (int64_t *)malloc(sizeof(int64_t) * (size_t)E);
        if (!next) return OR_EINVAL;
        for (int64_t e = 0; e < E; ++e) next[e] = group_offsets[e];
        for (int64_t f = 0; f < n_pairs; ++f) {
            int64_t r = next[topk_idx[f]]++;
            if (sorted_token_idx) sorted_token_idx[r] = (int32_t)(f / k);
            if (sorted_row_weight) sorted_row_weight[r] = topk_w ? topk_w[f] : 1.0f;
            if (token_topk_to_pos) token_topk_to_pos[f] = (int32_t)r;
        }
        free(next);
    }
    return OR_OK;
}

/* [CSDN "forward"] step 3: stacked_expert_tokens[r] = x_flat[token index of row r] */
int oracle_gather_rows(const void *x, const int32_t *sorted_token_idx, int64_t n_rows,
                       int64_t T, int64_t d_h, int dtype, void *a_out)
{
    oracle_init();
    if (!x || !sorted_token_idx || !a_out || n_rows < 0 || d_h <= 0 || !dtype_ok(dtype))
        return OR_EINVAL;
    size_t es = dtype == OR_F32 ? 4 : 2;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t t = sorted_token_idx[r];
        if (t < 0 || t >= T) return OR_EINVAL;
        memcpy((char *)a_out + (size_t)(r * d_h) * es, (const char *)x + (size_t)(t * d_h) * es,
               (size_t)d_h * es);
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* o4: the two grouped GEMM stages, block by block as the kernels walk them.   */
/* ------------------------------------------------------------------------- */

/* SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)), exact math in double. */
static double silu_d(double z) { return z / (1.0 + exp(-z)); }

/* Stage 1 for one row: h[rh, :] = rt(silu(A[ra] W_gate[g]^T) * (A[ra] W_up[g]^T)). */
static void stage1_row(const void *a, int64_t ra, const void *w_gate, const void *w_up, int64_t g,
                       int64_t d_h, int64_t d_e, int dtype, void *h, int64_t rh)
{
    for (int64_t n = 0; n < d_e; ++n) {
        const int64_t wrow = (g * d_e + n) * d_h;
        float gate = 0.0f, up = 0.0f;
        for (int64_t j = 0; j < d_h; ++j) {
            float av = load_elem(a, ra * d_h + j, dtype);
            gate = gate + av * load_elem(w_gate, wrow + j, dtype);
            up = up + av * load_elem(w_up, wrow + j, dtype);
        }
        float s = (float)silu_d((double)gate);
        float hv = s * up;
        store_elem(h, rh * d_e + n, dtype, hv);
    }
}

/* Stage 2 for one row: y[ry, :] = rt((h[rh] W_down[g]^T) * rw). */
static void stage2_row(const void *h, int64_t rh, const void *w_down, int64_t g, int64_t d_h,
                       int64_t d_e, int dtype, const float *rw, void *y, int64_t ry)
{
    for (int64_t o = 0; o < d_h; ++o) {
        const int64_t wrow = (g * d_h + o) * d_e;
        float acc = 0.0f;
        for (int64_t j = 0; j < d_e; ++j)
            acc = acc + load_elem(h, rh * d_e + j, dtype) * load_elem(w_down, wrow + j, dtype);
        if (rw) acc = acc * (*rw);
        store_elem(y, ry * d_h + o, dtype, acc);
    }
}

typedef struct {
    const void *a, *w1, *w2; /* stage 1: a, w_gate, w_up; stage 2: h, w_down */
    const int32_t *sizes, *offsets, *padded, *gidx;
    const float *row_weights;
    int64_t block_m, n_rows, d_h, d_e, E; int dtype; void *out;
    int stage;
} gemm_ctx;

/*
 * [CSDN stage-1 kernel] / [SKEL moe_routed_kernel first T.Kernel]: for block bx
 *   g = group_idx_for_bx[bx]
 *   m_start = bx*block - group_padded_offsets[g] + group_offsets[g]
 *   actual_rows = max(0, min(block, group_sizes[g] - (bx*block - group_padded_offsets[g])))
 *   gate = A[m_start:+rows] @ W_gate[g]^T, up = A @ W_up[g]^T  (fp32 accumulators)
 *   h = silu(gate) * up, rows i < actual_rows written, in the activation dtype.
 * The fp32 sum runs in ascending j.  silu is exact math, rounded to fp32 as
 * the page keeps it in the fp32 fragment; the product with up is fp32; h is
 * rounded once to the dtype.
 *
 * [CSDN stage-2 kernel] / [SKEL second T.Kernel]: same lookup,
 *   out = h[m_start:+rows] @ W_down[g]^T (fp32, ascending i), times
 *   RowWeights[m_start + i] when row weights are given, rounded to the dtype.
 */
static void gemm_blocks(int64_t lo, int64_t hi, void *vctx)
{
    gemm_ctx *c = (gemm_ctx *)vctx;
    const int64_t B = c->block_m;
    for (int64_t bx = lo; bx < hi; ++bx) {
        int64_t g = c->gidx[bx];
        int64_t m_start_padded = bx * B;
        int64_t m_start = m_start_padded - c->padded[g] + c->offsets[g];
        int64_t rows = c->sizes[g] - (m_start_padded - c->padded[g]);
        if (rows > B) rows = B;
        if (rows < 0) rows = 0;
        for (int64_t i = 0; i < rows; ++i) {
            int64_t r = m_start + i;
            if (c->stage == 1)
                stage1_row(c->a, r, c->w1, c->w2, g, c->d_h, c->d_e, c->dtype, c->out, r);
            else
                stage2_row(c->a, r, c->w1, g, c->d_h, c->d_e, c->dtype,
                           c->row_weights ? c->row_weights + r : NULL, c->out, r);
        }
    }
}

/* Per-row forms of the two stages for sampled checks of large problems: row i
 * of the inputs belongs to expert row_expert[i]; same arithmetic as above. */
typedef struct {
    const void *in, *w1, *w2; const int32_t *row_expert; const float *rw;
    int64_t d_h, d_e; int dtype; void *out; int stage;
} rows_ctx;

static void rows_range(int64_t lo, int64_t hi, void *vctx)
{
    rows_ctx *c = (rows_ctx *)vctx;
    for (int64_t i = lo; i < hi; ++i) {
        if (c->stage == 1)
            stage1_row(c->in, i, c->w1, c->w2, c->row_expert[i], c->d_h, c->d_e, c->dtype, c->out, i);
        else
            stage2_row(c->in, i, c->w1, c->row_expert[i], c->d_h, c->d_e, c->dtype,
                       c->rw ? c->rw + i : NULL, c->out, i);
    }
}

int oracle_rows_gate_up_silu(const void *a_rows, const int32_t *row_expert, int64_t n,
                             const void *w_gate, const void *w_up, int64_t d_h, int64_t d_e,
                             int64_t E, int dtype, void *h_rows, int nthreads)
{
    oracle_init();
    if (!a_rows || !row_expert || !w_gate || !w_up || !h_rows || n < 0 || d_h <= 0 ||
        d_e <= 0 || !dtype_ok(dtype))
        return OR_EINVAL;
    for (int64_t i = 0; i < n; ++i)
        if (row_expert[i] < 0 || row_expert[i] >= E) return OR_EINVAL;
    rows_ctx c = {a_rows, w_gate, w_up, row_expert, NULL, d_h, d_e, dtype, h_rows, 1};
    parallel_for(n, nthreads, rows_range, &c);
    return OR_OK;
}

int oracle_rows_down(const void *h_rows, const int32_t *row_expert, int64_t n, const void *w_down,
                     const float *row_weights, int64_t d_h, int64_t d_e, int64_t E, int dtype,
                     void *y_rows, int nthreads)
{
    oracle_init();
    if (!h_rows || !row_expert || !w_down || !y_rows || n < 0 || d_h <= 0 || d_e <= 0 ||
        !dtype_ok(dtype))
        return OR_EINVAL;
    for (int64_t i = 0; i < n; ++i)
        if (row_expert[i] < 0 || row_expert[i] >= E) return OR_EINVAL;
    rows_ctx c = {h_rows, w_down, NULL, row_expert, row_weights, d_h, d_e, dtype, y_rows, 2};
    parallel_for(n, nthreads, rows_range, &c);
    return OR_OK;
}

static int check_tables(const int32_t *sizes, const int32_t *offsets, const int32_t *padded,
                        const int32_t *gidx, int64_t m_blocks, int64_t n_rows, int64_t E,
                        int64_t block_m)
{
    if (!sizes || !offsets || !padded || !gidx || m_blocks < 0 || E <= 0 || block_m <= 0)
        return 0;
    for (int64_t bx = 0; bx < m_blocks; ++bx) {
        int64_t g = gidx[bx];
        if (g < 0 || g >= E) return 0;
        int64_t m_start = bx * block_m - padded[g] + offsets[g];
        int64_t rows = sizes[g] - (bx * block_m - padded[g]);
        if (rows > block_m) rows = block_m;
        if (rows > 0 && (m_start < 0 || m_start + rows > n_rows)) return 0;
    }
    return 1;
}

int oracle_grouped_gate_up_silu(const void *a, const void *w_gate, const void *w_up,
                                const int32_t *group_sizes, const int32_t *group_offsets,
                                const int32_t *group_padded_offsets,
                                const int32_t *group_idx_for_bx, int64_t m_blocks,
                                int64_t block_m, int64_t n_rows, int64_t d_h, int64_t d_e,
                                int64_t E, int dtype, void *h, int nthreads)
{
    oracle_init();
    if (!a || !w_gate || !w_up || !h || d_h <= 0 || d_e <= 0 || !dtype_ok(dtype) ||
        !check_tables(group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                      m_blocks, n_rows, E, block_m))
        return OR_EINVAL;
    gemm_ctx c = {a, w_gate, w_up, group_sizes, group_offsets, group_padded_offsets,
                  group_idx_for_bx, NULL, block_m, n_rows, d_h, d_e, E, dtype, h, 1};
    parallel_for(m_blocks, nthreads, gemm_blocks, &c);
    return OR_OK;
}

int oracle_grouped_down(const void *h, const void *w_down, const int32_t *group_sizes,
                        const int32_t *group_offsets, const int32_t *group_padded_offsets,
                        const int32_t *group_idx_for_bx, int64_t m_blocks, int64_t block_m,
                        const float *row_weights, int64_t n_rows, int64_t d_h, int64_t d_e,
                        int64_t E, int dtype, void *y, int nthreads)
{
    oracle_init();
    if (!h || !w_down || !y || d_h <= 0 || d_e <= 0 || !dtype_ok(dtype) ||
        !check_tables(group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                      m_blocks, n_rows, E, block_m))
        return OR_EINVAL;
    gemm_ctx c = {h, w_down, NULL, group_sizes, group_offsets, group_padded_offsets,
                  group_idx_for_bx, row_weights, block_m, n_rows, d_h, d_e, E, dtype, y, 2};
    parallel_for(m_blocks, nthreads, gemm_blocks, &c);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* o4q: the expert MLP with int4 weights (weight-only, W4A16).                 */
/* ------------------------------------------------------------------------- */
/*
 * [SKEL w4a8_dequant_gemm]: the weight is int4, two values per uint8 byte;
 * element j of a row sits in byte j / 2, nibble j % 2 counted from the low
 * end, and is sign-extended (two's complement, -8 .. 7) when unpacked on
 * chip; the unpacked value is cast to the compute type and fed to the GEMM.
 * [SKEL quantisation notes]: weight-only W4A16 is the same kernel with
 * 16-bit activations.  Reading (the pages print no scale): an optional fp32
 * scale per output channel multiplies the fp32 sum (NULL = the plain int4
 * value), i.e. for stage 1
 *   G = (sum_j a_j * q_gate[g,n,j]) * s_gate[g,n],  U likewise with s_up,
 *   h = rt(silu(G) * U)
 * and for stage 2  y = rt((sum_i h_i * q_down[g,o,i]) * s_down[g,o] (* rw)).
 * Every product a * q is exact in fp32; sums in ascending index.
 */
void oracle_unpack_int4(const uint8_t *packed, int64_t n, int8_t *out)
{
    for (int64_t j = 0; j < n; ++j) {
        const int nib = (packed[j / 2] >> (4 * (int)(j % 2))) & 0xF;
        out[j] = (int8_t)(nib >= 8 ? nib - 16 : nib);
    }
}

typedef struct {
    const void *a; const int8_t *q1, *q2; const float *s1, *s2;
    const int32_t *sizes, *offsets, *padded, *gidx;
    const float *row_weights;
    int64_t block_m, n_rows, d_h, d_e, E; int dtype; void *out;
    int stage;
} gemm_q_ctx;

static void stage1_row_q(const gemm_q_ctx *c, int64_t r, int64_t g)
{
    for (int64_t n = 0; n < c->d_e; ++n) {
        const int64_t wrow = (g * c->d_e + n) * c->d_h;
        float gate = 0.0f, up = 0.0f;
        for (int64_t j = 0; j < c->d_h; ++j) {
            float av = load_elem(c->a, r * c->d_h + j, c->dtype);
            gate = gate + av * (float)c->q1[wrow + j];
            up = up + av * (float)c->q2[wrow + j];
        }
        if (c->s1) gate = gate * c->s1[g * c->d_e + n];
        if (c->s2) up = up * c->s2[g * c->d_e + n];
        float sv = (float)silu_d((double)gate);
        store_elem(c->out, r * c->d_e + n, c->dtype, sv * up);
    }
}

static void stage2_row_q(const gemm_q_ctx *c, int64_t r, int64_t g)
{
    for (int64_t o = 0; o < c->d_h; ++o) {
        const int64_t wrow = (g * c->d_h + o) * c->d_e;
        float acc = 0.0f;
        for (int64_t j = 0; j < c->d_e; ++j)
            acc = acc + load_elem(c->a, r * c->d_e + j, c->dtype) * (float)c->q1[wrow + j];
        if (c->s1) acc = acc * c->s1[g * c->d_h + o];
        if (c->row_weights) acc = acc * c->row_weights[r];
        store_elem(c->out, r * c->d_h + o, c->dtype, acc);
    }
}

/* the block walk of the CSDN stage kernels (see gemm_blocks), int4 weights */
static void gemm_q_blocks(int64_t lo, int64_t hi, void *vctx)
{
    gemm_q_ctx *c = (gemm_q_ctx *)vctx;
    const int64_t B = c->block_m;
    for (int64_t bx = lo; bx < hi; ++bx) {
        int64_t g = c->gidx[bx];
        int64_t m_start = bx * B - c->padded[g] + c->offsets[g];
        int64_t rows = c->sizes[g] - (bx * B - c->padded[g]);
        if (rows > B) rows = B;
        if (rows < 0) rows = 0;
        for (int64_t i = 0; i < rows; ++i) {
            if (c->stage == 1) stage1_row_q(c, m_start + i, g);
            else stage2_row_q(c, m_start + i, g);
        }
    }
}

/* q_gate, q_up: [E, d_e, d_h / 2] packed bytes; s_gate, s_up: [E, d_e] or NULL */
int oracle_grouped_gate_up_silu_w4(const void *a, const uint8_t *q_gate, const uint8_t *q_up,
                                   const float *s_gate, const float *s_up,
                                   const int32_t *group_sizes, const int32_t *group_offsets,
                                   const int32_t *group_padded_offsets,
                                   const int32_t *group_idx_for_bx, int64_t m_blocks,
                                   int64_t block_m, int64_t n_rows, int64_t d_h, int64_t d_e,
                                   int64_t E, int dtype, void *h, int nthreads)
{
    oracle_init();
    if (!a || !q_gate || !q_up || !h || d_h <= 0 || d_h % 2 != 0 || d_e <= 0 ||
        (dtype != 0 && dtype != 1) ||
        !check_tables(group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                      m_blocks, n_rows, E, block_m))
        return OR_EINVAL;
    const int64_t n = E * d_e * d_h;
    int8_t *qg = (int8_t *)malloc((size_t)n), *qu = (int8_t *)malloc((size_t)n);
    if (!qg || !qu) { free(qg); free(qu); return OR_EINVAL; }
    oracle_unpack_int4(q_gate, n, qg);
    oracle_unpack_int4(q_up, n, qu);
    gemm_q_ctx c = {a, qg, qu, s_gate, s_up, group_sizes, group_offsets, group_padded_offsets,
                    group_idx_for_bx, NULL, block_m, n_rows, d_h, d_e, E, dtype, h, 1};
    parallel_for(m_blocks, nthreads, gemm_q_blocks, &c);
    free(qg);
    free(qu);
    return OR_OK;
}

/* q_down: [E, d_h, d_e / 2] packed bytes; s_down: [E, d_h] or NULL */
int oracle_grouped_down_w4(const void *h, const uint8_t *q_down, const float *s_down,
                           const int32_t *group_sizes, const int32_t *group_offsets,
                           const int32_t *group_padded_offsets, const int32_t *group_idx_for_bx,
                           int64_t m_blocks, int64_t block_m, const float *row_weights,
                           int64_t n_rows, int64_t d_h, int64_t d_e, int64_t E, int dtype,
                           void *y, int nthreads)
{
    oracle_init();
    if (!h || !q_down || !y || d_h <= 0 || d_e <= 0 || d_e % 2 != 0 || (dtype != 0 && dtype != 1) ||
        !check_tables(group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                      m_blocks, n_rows, E, block_m))
        return OR_EINVAL;
    const int64_t n = E * d_h * d_e;
    int8_t *qd = (int8_t *)malloc((size_t)n);
    if (!qd) return OR_EINVAL;
    oracle_unpack_int4(q_down, n, qd);
    gemm_q_ctx c = {h, qd, NULL, s_down, NULL, group_sizes, group_offsets, group_padded_offsets,
                    group_idx_for_bx, row_weights, block_m, n_rows, d_h, d_e, E, dtype, y, 2};
    parallel_for(m_blocks, nthreads, gemm_q_blocks, &c);
    free(qd);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* f3: W4A8 -- int4 weights x int8 activations, int32 sums.                   */
/* ------------------------------------------------------------------------- */
/*
 * [SKEL w4a8_dequant_gemm]: A int8 [M, K]; B uint8 [N, K / 2] in the int4
 * format above; every int4 value is sign-extended to int8 on chip and the
 * product summed in an int32 accumulator; the result is written transposed:
 *   Ct[n, m] = sum_k A[m, k] * int4(B)[n, k]        (Ct int32 [N, M]).
 * [SKEL quantisation notes]: weight + activation quantisation (W4A8); the
 * skeleton returns the raw int32 sums (the dequantisation scales are the
 * caller's).  The sum is formed here in int64: |Ct| <= 8 * 128 * K, so for
 * K <= 2^20 an int32 accumulator cannot wrap and the two agree (larger K is
 * refused).
 */
#define W4A8_MAX_K (1LL << 20)

static int64_t dot_w4a8(const int8_t *a, const uint8_t *brow, int64_t K)
{
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k) {
        const int nib = (brow[k / 2] >> (4 * (int)(k % 2))) & 0xF;
        acc += (int64_t)a[k] * (int64_t)(nib >= 8 ? nib - 16 : nib);
    }
    return acc;
}

typedef struct {
    const int8_t *a; const uint8_t *b; int64_t M, N, K; int32_t *ct;
} w4a8_ctx;

static void w4a8_cols(int64_t lo, int64_t hi, void *vctx)
{
    w4a8_ctx *c = (w4a8_ctx *)vctx;
    for (int64_t n = lo; n < hi; ++n)
        for (int64_t m = 0; m < c->M; ++m)
            c->ct[n * c->M + m] = (int32_t)dot_w4a8(c->a + m * c->K, c->b + n * (c->K / 2), c->K);
}

int oracle_gemm_w4a8(const int8_t *A, const uint8_t *B, int64_t M, int64_t N, int64_t K, int32_t *Ct,
                     int nthreads)
{
    if (!A || !B || !Ct || M <= 0 || N <= 0 || K <= 0 || K % 2 != 0 || K > W4A8_MAX_K) return OR_EINVAL;
    w4a8_ctx c = {A, B, M, N, K, Ct};
    parallel_for(N, nthreads, w4a8_cols, &c);
    return OR_OK;
}

/*
 * The grouped form for the routed experts: the block walk of [SKEL
 * moe_routed_kernel] / [CSDN stage 2 down] over the dispatch tables, each
 * block's rows multiplied by its expert's int4 weight:
 *   C[r, n] = sum_k a[r, k] * int4(B[g])[n, k]   (a int8 [n_rows, K] in
 *   expert order, B [E, N, K / 2], C int32 [n_rows, N], g the row's expert).
 */
typedef struct {
    const int8_t *a; const uint8_t *b;
    const int32_t *sizes, *offsets, *padded, *gidx;
    int64_t block_m, N, K; int32_t *c;
} w4a8_grouped_ctx;

static void w4a8_blocks(int64_t lo, int64_t hi, void *vctx)
{
    w4a8_grouped_ctx *c = (w4a8_grouped_ctx *)vctx;
    const int64_t B = c->block_m;
    for (int64_t bx = lo; bx < hi; ++bx) {
        const int64_t g = c->gidx[bx];
        const int64_t m_start = bx * B - c->padded[g] + c->offsets[g];
        int64_t rows = c->sizes[g] - (bx * B - c->padded[g]);
        if (rows > B) rows = B;
        if (rows < 0) rows = 0;
        for (int64_t i = 0; i < rows; ++i) {
            const int64_t r = m_start + i;
            for (int64_t n = 0; n < c->N; ++n)
                c->c[r * c->N + n] =
                    (int32_t)dot_w4a8(c->a + r * c->K, c->b + (g * c->N + n) * (c->K / 2), c->K);
        }
    }
}

int oracle_grouped_gemm_w4a8(const int8_t *a, const uint8_t *B, const int32_t *group_sizes,
                             const int32_t *group_offsets, const int32_t *group_padded_offsets,
                             const int32_t *group_idx_for_bx, int64_t m_blocks, int64_t block_m,
                             int64_t n_rows, int64_t N, int64_t K, int64_t E, int32_t *C, int nthreads)
{
    if (!a || !B || !C || N <= 0 || K <= 0 || K % 2 != 0 || K > W4A8_MAX_K ||
        !check_tables(group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                      m_blocks, n_rows, E, block_m))
        return OR_EINVAL;
    w4a8_grouped_ctx c = {a, B, group_sizes, group_offsets, group_padded_offsets, group_idx_for_bx,
                          block_m, N, K, C};
    parallel_for(m_blocks, nthreads, w4a8_blocks, &c);
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* o5: moe_reduce_fused.                                                       */
/* ------------------------------------------------------------------------- */
/*
 * [PR55 section 1]: one output row per token t; for the K slots in ascending
 * order, skip pos < 0 (padding), otherwise add topk_weights[t,k] *
 * x[pos[t,k], :] into an fp32 accumulator; cast once to the output dtype.
 * Without weights every slot has weight 1.  A pos >= n_rows or < -1 is not a
 * case the page covers: it is skipped and reported through *err_flag.
 * The accumulation is acc = acc + w * x with a separate rounding of w * x.
 */
typedef struct {
    const void *x; int64_t n_rows; const int32_t *pos; const float *w;
    const float *x_sf, *sf;
    int64_t K, H; int in_dtype, out_dtype; void *out; int bad;
} reduce_ctx;

static void reduce_rows(int64_t lo, int64_t hi, void *vctx)
{
    reduce_ctx *c = (reduce_ctx *)vctx;
    float *acc = (float *)malloc(sizeof(float) * (size_t)c->H);
    for (int64_t t = lo; t < hi; ++t) {
        for (int64_t hh = 0; hh < c->H; ++hh) acc[hh] = 0.0f;
        for (int64_t k = 0; k < c->K; ++k) {
            int64_t p = c->pos[t * c->K + k];
            if (p < 0 || p >= c->n_rows) {
                if (p < -1 || p >= c->n_rows) __atomic_store_n(&c->bad, 1, __ATOMIC_RELAXED);
                continue;
            }
            float w = c->w ? c->w[t * c->K + k] : 1.0f;
            if (c->x_sf) w = w * c->x_sf[p];          /* one multiply per routed slot */
            for (int64_t hh = 0; hh < c->H; ++hh) {
                float prod = w * load_elem(c->x, p * c->H + hh, c->in_dtype);
                acc[hh] = acc[hh] + prod;
            }
        }
        float s = c->sf ? c->sf[t] : 1.0f;
        for (int64_t hh = 0; hh < c->H; ++hh) {
            float v = c->sf ? acc[hh] * s : acc[hh];  /* one multiply per output element */
            store_elem(c->out, t * c->H + hh, c->out_dtype, v);
        }
    }
    free(acc);
}

/*
 * [PR55 section 1, variants]: the same combine with the compile-time switches
 * of the page's four ops: x_sf (WithXsf), a scale per expanded row of x, is
 * folded into the slot weight (w * x_sf[pos], one multiply per routed slot);
 * sf (Quantized), read here as one scale per token, multiplies every output
 * element of that token after the sum (one multiply per output element);
 * the output may be float8 e4m3fn (Fp8 / Quantized), rounded to nearest even
 * and saturated to +-448.
 */
int oracle_reduce_fused_scaled(const void *x, int64_t n_rows, const int32_t *token_topk_to_pos,
                               const float *topk_weights, const float *x_sf, const float *sf,
                               int64_t T, int64_t K, int64_t H, int in_dtype, int out_dtype,
                               void *out, int32_t *err_flag, int nthreads)
{
    oracle_init();
    if (!out || !token_topk_to_pos || T < 0 || K <= 0 || H <= 0 || n_rows < 0 ||
        (!x && n_rows > 0) || !dtype_ok(in_dtype) || !out_dtype_ok(out_dtype))
        return OR_EINVAL;
    reduce_ctx c = {x, n_rows, token_topk_to_pos, topk_weights, x_sf, sf, K, H, in_dtype,
                    out_dtype, out, 0};
    parallel_for(T, nthreads, reduce_rows, &c);
    if (err_flag) *err_flag = c.bad;
    return OR_OK;
}

int oracle_reduce_fused(const void *x, int64_t n_rows, const int32_t *token_topk_to_pos,
                        const float *topk_weights, int64_t T, int64_t K, int64_t H,
                        int in_dtype, int out_dtype, void *out, int32_t *err_flag,
                        int nthreads)
{
    if (!dtype_ok(out_dtype)) return OR_EINVAL;
    return oracle_reduce_fused_scaled(x, n_rows, token_topk_to_pos, topk_weights, NULL, NULL, T,
                                      K, H, in_dtype, out_dtype, out, err_flag, nthreads);
}

/* ------------------------------------------------------------------------- */
/* o6: dense per-token brute force (no dispatch tables at all).               */
/* ------------------------------------------------------------------------- */
/*
 * For each listed token t and each slot j in ascending order, run expert
 * e = topk_idx[t, j] directly on x[t]: h = rt(silu(x W_gate[e]^T) * (x W_up[e]^T)),
 * y = rt(h W_down[e]^T), acc += topk_w[t, j] * y, then out = rt(acc).  The
 * arithmetic per element is the same as stages 1 and 2 plus the combine, so it
 * equals their composition through the dispatch tables bit for bit.
 */
typedef struct {
    const void *x, *w_gate, *w_up, *w_down; const int32_t *topk_idx; const float *topk_w;
    const int32_t *tokens; int64_t d_h, d_e, k; int dtype; void *out;
} dense_ctx;

static void dense_tokens(int64_t lo, int64_t hi, void *vctx)
{
    dense_ctx *c = (dense_ctx *)vctx;
    float *xv = (float *)malloc(sizeof(float) * (size_t)c->d_h);
    float *hv = (float *)malloc(sizeof(float) * (size_t)c->d_e);
    float *acc = (float *)malloc(sizeof(float) * (size_t)c->d_h);
    for (int64_t s = lo; s < hi; ++s) {
        int64_t t = c->tokens[s];
        for (int64_t j = 0; j < c->d_h; ++j) xv[j] = load_elem(c->x, t * c->d_h + j, c->dtype);
        for (int64_t o = 0; o < c->d_h; ++o) acc[o] = 0.0f;
        for (int64_t slot = 0; slot < c->k; ++slot) {
            int64_t e = c->topk_idx[t * c->k + slot];
            float w = c->topk_w[t * c->k + slot];
            for (int64_t n = 0; n < c->d_e; ++n) {
                const int64_t wrow = (e * c->d_e + n) * c->d_h;
                float gate = 0.0f, up = 0.0f;
                for (int64_t j = 0; j < c->d_h; ++j) {
                    gate = gate + xv[j] * load_elem(c->w_gate, wrow + j, c->dtype);
                    up = up + xv[j] * load_elem(c->w_up, wrow + j, c->dtype);
                }
                float sg = (float)silu_d((double)gate);
                float hval = sg * up;
                /* round-trip through the storage dtype, as h is stored */
                uint16_t tmp16; float tmp32;
                if (c->dtype == OR_F32) { tmp32 = hval; hv[n] = tmp32; }
                else { store_elem(&tmp16, 0, c->dtype, hval); hv[n] = load_elem(&tmp16, 0, c->dtype); }
            }
            for (int64_t o = 0; o < c->d_h; ++o) {
                const int64_t wrow = (e * c->d_h + o) * c->d_e;
                float yacc = 0.0f;
                for (int64_t n = 0; n < c->d_e; ++n)
                    yacc = yacc + hv[n] * load_elem(c->w_down, wrow + n, c->dtype);
                float yv;
                if (c->dtype == OR_F32) yv = yacc;
                else { uint16_t tmp16; store_elem(&tmp16, 0, c->dtype, yacc); yv = load_elem(&tmp16, 0, c->dtype); }
                float prod = w * yv;
                acc[o] = acc[o] + prod;
            }
        }
        for (int64_t o = 0; o < c->d_h; ++o) store_elem(c->out, s * c->d_h + o, c->dtype, acc[o]);
    }
    free(xv); free(hv); free(acc);
}

int oracle_moe_tokens_dense(const void *x, const void *w_gate, const void *w_up,
                            const void *w_down, const int32_t *topk_idx, const float *topk_w,
                            const int32_t *tokens, int64_t n_tokens, int64_t T, int64_t d_h,
                            int64_t d_e, int64_t E, int64_t k, int dtype, void *out,
                            int nthreads)
{
    oracle_init();
    if (!x || !w_gate || !w_up || !w_down || !topk_idx || !topk_w || !tokens || !out ||
        d_h <= 0 || d_e <= 0 || E <= 0 || k <= 0 || !dtype_ok(dtype))
        return OR_EINVAL;
    for (int64_t s = 0; s < n_tokens; ++s) {
        if (tokens[s] < 0 || tokens[s] >= T) return OR_EINVAL;
        for (int64_t j = 0; j < k; ++j) {
            int32_t e = topk_idx[tokens[s] * k + j];
            if (e < 0 || e >= E) return OR_EINVAL;
        }
    }
    dense_ctx c = {x, w_gate, w_up, w_down, topk_idx, topk_w, tokens, d_h, d_e, k, dtype, out};
    parallel_for(n_tokens, nthreads, dense_tokens, &c);
    return OR_OK;
}

/*
 * CPU oracle for the next-scale VAR attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so and
 * called by the test-suite, the smoke check and the benchmark's CPU-baseline
 * leg.  The CUDA library never links, includes or calls it, and it shares no
 * code with the CUDA library.
 *
 * Everything is plain fp64 loops over the exact bf16 input values (widened to
 * double), in the order the method states, parallelised only over independent
 * output rows.  Sources (page titles; sections/equations):
 *
 *  - Dense cross-scale attention: "SparVAR: Exploring Sparsity in Visual
 *    AutoRegressive Modeling" (abstract): at each next-scale step the queries
 *    of the current grid attend to all tokens of all earlier scales (and the
 *    current one, through the KV cache of "ARVAR", Background & Motivation).
 *  - Block-sparse attention: SparVAR abstract -- attention sinks plus
 *    cross-scale local windows, evaluated block-wise.
 *  - Pivot selection: "FastVAR: Linear Visual Autoregressive Modeling via
 *    Cached Token Pruning" (abstract: forward only pivotal tokens) and ARVAR
 *    Key Design 2 (Top-K indices used to gather).  The score is
 *    ||x_i - mean_grid(x)||_2, the token's distance from the grid mean (its DC
 *    component): a frequency-style criterion, as ARVAR's Related Work
 *    describes FastVAR's selection.
 *  - Restore + scatter: ARVAR Key Design 3, Eq. (8)-(9):
 *    Y_T = Scatter(Up(Y_{T-N}; h_T, w_T), I_T, Yhat_T), scatter overwrites.
 *  - Dynamic sparse pattern: SparVAR abstract -- the sparse attention pattern
 *    of later high-resolution scales is predicted from a sparse decision
 *    scale.  This file gives the attention mass each unit of keys receives
 *    from each decision-step query (oracle_unit_mass) and attention under an
 *    explicit token-level keep mask (oracle_attention_keep); the selection and
 *    index mapping built on them are in __init__.py.
 *
 * Readings taken where the pages are silent:
 *  - no causal mask inside a step; softmax scale 1/sqrt(head_dim);
 *  - the softmax subtracts the row maximum (identical in exact arithmetic);
 *  - pivot score ranked by the squared distance, evaluated in fp64 as a
 *    pairwise-halving tree over channels; ties go to the lower flat index;
 *    selected indices returned in ascending order;
 *  - bilinear upsampling with half-pixel centres, edge clamp, no antialias;
 *  - block mask: the query block's +-radius block window, rescaled into each
 *    key scale's grid and rounded outward to that scale's blocks; scales with
 *    side <= sink_max_side are kept whole (attention sinks).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (see build.py).
 * -ffp-contract=off keeps a*b+c as two rounded operations, as written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_SCALES 32

/* Threads the parallel loops below use (for reporting CPU-baseline timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Block mask (SparVAR: sinks + cross-scale local window)              */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t n_scales;
    int32_t side[ORACLE_MAX_SCALES];
    int32_t step;            /* query scale index                      */
    int32_t qblock_side;     /* query block = qblock_side^2 patch      */
    int32_t radius;          /* window half-width, in query blocks     */
    int32_t sink_max_side;   /* scales with side <= this: always kept  */
} oracle_mask_spec;

/* One axis of the window rule.  qb: query block coordinate on this axis;
 * t: key coordinate on this axis inside a scale of side s; sq: query side. */
static int axis_in_window(const oracle_mask_spec* m, int qb, int t, int s)
{
    const long sq = m->side[m->step];
    const long bs = m->qblock_side;
    long lo = bs * (long)(qb - m->radius);
    long hi = bs * (long)(qb + m->radius + 1);
    if (lo < 0) lo = 0;
    if (hi > sq) hi = sq;
    /* rescale the window into the key scale, rounding outward */
    long lo_s = (lo * s) / sq;
    long hi_s = (hi * s + sq - 1) / sq;
    /* the key's own block in its scale */
    long b0 = (t / bs) * bs;
    long b1 = b0 + bs;
    if (b1 > s) b1 = s;
    return b0 < hi_s && lo_s < b1;
}

/* 1 if query token qi (flat index in the query grid) keeps flat cache key j. */
static int key_kept(const oracle_mask_spec* m, int qi, int j)
{
    const int sq = m->side[m->step];
    const int qy = qi / sq, qx = qi % sq;
    const int by = qy / m->qblock_side, bx = qx / m->qblock_side;
    int off = 0;
    for (int sc = 0; sc <= m->step; sc++) {
        const int s = m->side[sc];
        const int n = s * s;
        if (j < off + n) {
            if (s <= m->sink_max_side) return 1;
            const int r = (j - off) / s, c = (j - off) % s;
            return axis_in_window(m, by, r, s) && axis_in_window(m, bx, c, s);
        }
        off += n;
    }
    return 0;
}

/* Token-level mask rows for query tokens [q0, q1): out[(qi-q0)*L + j]. */
int oracle_block_mask_rows(const oracle_mask_spec* m, int q0, int q1, uint8_t* out)
{
    if (!m || m->step < 0 || m->step >= m->n_scales || m->qblock_side <= 0) return 1;
    int L = 0;
    for (int sc = 0; sc <= m->step; sc++) L += m->side[sc] * m->side[sc];
#pragma omp parallel for schedule(static)
    for (int qi = q0; qi < q1; qi++)
        for (int j = 0; j < L; j++) out[(size_t)(qi - q0) * L + j] = (uint8_t)key_kept(m, qi, j);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Attention                                                           */
/* ------------------------------------------------------------------ */

/* One output row: o = sum_j softmax_j(q.k_j * scale) v_j over kept keys.
 * sbuf holds L doubles.  An empty key set gives a zero row. */
static void attend_row(int L, int D, double scale, const uint16_t* q, const uint16_t* K,
                       const uint16_t* V, const oracle_mask_spec* m, const uint8_t* keep_row, int qi,
                       double* sbuf, double* out)
{
    double mx = -INFINITY;
    for (int j = 0; j < L; j++) {
        if ((m && !key_kept(m, qi, j)) || (keep_row && !keep_row[j])) { sbuf[j] = -INFINITY; continue; }
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += bf16_to_f64(q[d]) * bf16_to_f64(K[(size_t)j * D + d]);
        sbuf[j] = dot * scale;
        if (sbuf[j] > mx) mx = sbuf[j];
    }
    for (int d = 0; d < D; d++) out[d] = 0.0;
    if (mx == -INFINITY) return;
    double l = 0.0;
    for (int j = 0; j < L; j++) {
        if (sbuf[j] == -INFINITY) continue;
        const double p = exp(sbuf[j] - mx);
        l += p;
        for (int d = 0; d < D; d++) out[d] += p * bf16_to_f64(V[(size_t)j * D + d]);
    }
    for (int d = 0; d < D; d++) out[d] /= l;
}

/*
 * Attention of step queries over the first L cached keys.
 *   q: [B][H][N][D] bf16 bits;  k, v: [B][H][kv_cap][D] bf16 bits (first L rows used)
 *   rows: n_rows flat query ids ((b*H + h)*N + i), or NULL for all B*H*N rows
 *   mask: NULL for dense, else the block-sparse rule
 *   o: [n_rows][D] (or [B*H*N][D]) doubles
 */
int oracle_attention(int B, int H, int N, int L, int kv_cap, int D, double scale,
                     const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     long n_rows, const int64_t* rows, const oracle_mask_spec* m, double* o)
{
    if (B <= 0 || H <= 0 || N < 0 || L <= 0 || D <= 0 || kv_cap < L) return 1;
    const long total = rows ? n_rows : (long)B * H * N;
    int bad = 0;
#pragma omp parallel
    {
        double* sbuf = (double*)malloc(sizeof(double) * (size_t)L);
        if (!sbuf) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long r = 0; r < total; r++) {
                const long flat = rows ? rows[r] : r;
                if (flat < 0 || flat >= (long)B * H * N) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                const long bh = flat / N;
                const int qi = (int)(flat % N);
                attend_row(L, D, scale, q + (size_t)flat * D, k + (size_t)bh * kv_cap * D,
                           v + (size_t)bh * kv_cap * D, m, NULL, qi, sbuf, o + (size_t)r * D);
            }
            free(sbuf);
        }
    }
    return bad;
}

/*
 * As oracle_attention (all rows), with the kept keys given token by token:
 * query i of every (b, h) attends to key j < L iff keep[i * L + j] != 0.
 */
int oracle_attention_keep(int B, int H, int N, int L, int kv_cap, int D, double scale,
                          const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const uint8_t* keep, double* o)
{
    if (B <= 0 || H <= 0 || N < 0 || L <= 0 || D <= 0 || kv_cap < L || !keep) return 1;
    const long total = (long)B * H * N;
    int bad = 0;
#pragma omp parallel
    {
        double* sbuf = (double*)malloc(sizeof(double) * (size_t)L);
        if (!sbuf) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long r = 0; r < total; r++) {
                const long bh = r / N;
                const int qi = (int)(r % N);
                attend_row(L, D, scale, q + (size_t)r * D, k + (size_t)bh * kv_cap * D,
                           v + (size_t)bh * kv_cap * D, NULL, keep + (size_t)qi * L, qi, sbuf,
                           o + (size_t)r * D);
            }
            free(sbuf);
        }
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Attention retrospect (ARVAR Key Design 2): row statistics and the   */
/* probability each token of the source grid receives                  */
/* ------------------------------------------------------------------ */

/* s_j = q . k_j * scale for j < L; returns the maximum. */
static double row_scores(int L, int D, double scale, const uint16_t* q, const uint16_t* K, double* s)
{
    double mx = -INFINITY;
    for (int j = 0; j < L; j++) {
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += bf16_to_f64(q[d]) * bf16_to_f64(K[(size_t)j * D + d]);
        s[j] = dot * scale;
        if (s[j] > mx) mx = s[j];
    }
    return mx;
}

/*
 * lse[bh][i] = log2(sum_j e^(s_ij)), s_ij = q_i . k_j * scale over the first L
 * keys, so that the attention probability is 2^(s_ij log2(e) - lse_i).
 */
int oracle_attention_lse(int B, int H, int N, int L, int kv_cap, int D, double scale,
                         const uint16_t* q, const uint16_t* k, double* lse)
{
    if (B <= 0 || H <= 0 || N <= 0 || L <= 0 || D <= 0 || kv_cap < L) return 1;
    int bad = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        if (!s) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long flat = 0; flat < (long)B * H * N; flat++) {
                const long bh = flat / N;
                const double mx = row_scores(L, D, scale, q + (size_t)flat * D, k + (size_t)bh * kv_cap * D, s);
                double l = 0.0;
                for (int j = 0; j < L; j++) l += exp(s[j] - mx);
                lse[flat] = (mx + log(l)) / log(2.0);
            }
            free(s);
        }
    }
    return bad;
}

/*
 * sal[bh][j] = sum_i P[i, L - N + j]: the softmax probability (over all L keys)
 * that key L - N + j of the self block -- token j of the N-token source grid --
 * receives from each of the N source queries, summed over the queries.
 */
int oracle_saliency(int B, int H, int N, int L, int kv_cap, int D, double scale,
                    const uint16_t* q, const uint16_t* k, double* sal)
{
    if (B <= 0 || H <= 0 || N <= 0 || L < N || D <= 0 || kv_cap < L) return 1;
    int bad = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        if (!s) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(static)
            for (long bh = 0; bh < (long)B * H; bh++) {
                double* out = sal + (size_t)bh * N;
                for (int j = 0; j < N; j++) out[j] = 0.0;
                for (int i = 0; i < N; i++) {
                    const double mx = row_scores(L, D, scale, q + ((size_t)bh * N + i) * D,
                                                 k + (size_t)bh * kv_cap * D, s);
                    double l = 0.0;
                    for (int j = 0; j < L; j++) l += exp(s[j] - mx);
                    for (int j = 0; j < N; j++) out[j] += exp(s[L - N + j] - mx) / l;
                }
            }
            free(s);
        }
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Dynamic sparse pattern (SparVAR: a sparse decision scale)           */
/* ------------------------------------------------------------------ */

/*
 * mass[(bh * N + i) * U + u] = the softmax probability (over all L keys) that
 * query i of (b, h) gives to the keys j of unit u (unit_of[j] == u), summed:
 * the attention mass a unit of keys receives.  unit_of[j] in [0, U), j < L.
 */
int oracle_unit_mass(int B, int H, int N, int L, int kv_cap, int D, double scale,
                     const uint16_t* q, const uint16_t* k, const int32_t* unit_of, int U,
                     double* mass)
{
    if (B <= 0 || H <= 0 || N <= 0 || L <= 0 || D <= 0 || kv_cap < L || U <= 0 || !unit_of) return 1;
    for (int j = 0; j < L; j++)
        if (unit_of[j] < 0 || unit_of[j] >= U) return 1;
    int bad = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        if (!s) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(static)
            for (long r = 0; r < (long)B * H * N; r++) {
                const long bh = r / N;
                const double mx = row_scores(L, D, scale, q + (size_t)r * D, k + (size_t)bh * kv_cap * D, s);
                double l = 0.0;
                for (int j = 0; j < L; j++) l += exp(s[j] - mx);
                double* out = mass + (size_t)r * U;
                for (int u = 0; u < U; u++) out[u] = 0.0;
                for (int j = 0; j < L; j++) out[unit_of[j]] += exp(s[j] - mx) / l;
            }
            free(s);
        }
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Pivot score + top-K (FastVAR cached token pruning)                  */
/* ------------------------------------------------------------------ */

/* fp64 sum of t[0..n) as a pairwise-halving tree: left half first, split at n/2. */
static double tree_sum(const double* t, int n)
{
    if (n == 1) return t[0];
    const int h = n / 2;
    const double a = tree_sum(t, h);
    const double b = tree_sum(t + h, n - h);
    return a + b;
}

/* mean[b][c] = (sum_i x[b][i][c]) / N, summed sequentially over i in fp64. */
int oracle_pivot_mean(int B, int N, int C, const uint16_t* x, double* mean)
{
    if (B <= 0 || N <= 0 || C <= 0) return 1;
#pragma omp parallel for schedule(static)
    for (long bc = 0; bc < (long)B * C; bc++) {
        const long b = bc / C, c = bc % C;
        double s = 0.0;
        for (int i = 0; i < N; i++) s += bf16_to_f64(x[((size_t)b * N + i) * C + c]);
        mean[bc] = s / (double)N;
    }
    return 0;
}

/* score[b][i] = sum_c (x[b][i][c] - mean[b][c])^2, each term rounded, tree-summed. */
int oracle_pivot_scores(int B, int N, int C, const uint16_t* x, const double* mean, double* score)
{
    if (B <= 0 || N <= 0 || C <= 0) return 1;
    int bad = 0;
#pragma omp parallel
    {
        double* t = (double*)malloc(sizeof(double) * (size_t)C);
        if (!t) {
#pragma omp atomic write
            bad = 2;
        } else {
#pragma omp for schedule(static)
            for (long bi = 0; bi < (long)B * N; bi++) {
                const long b = bi / N;
                for (int c = 0; c < C; c++) {
                    const double d = bf16_to_f64(x[(size_t)bi * C + c]) - mean[b * C + c];
                    t[c] = d * d;
                }
                score[bi] = tree_sum(t, C);
            }
            free(t);
        }
    }
    return bad;
}

typedef struct { double s; int32_t i; } scored;

/* larger score first; equal scores: lower index first */
static int by_score_desc(const void* a, const void* b)
{
    const scored* x = (const scored*)a;
    const scored* y = (const scored*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->i > y->i) - (x->i < y->i);
}

static int by_int_asc(const void* a, const void* b)
{
    const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/*
 * Keep the K highest-scoring tokens of each batch element; idx[b][0..K) in
 * ascending order.  score (optional) receives [B][N] scores.
 */
int oracle_pivot_select(int B, int N, int C, const uint16_t* x, int K, int32_t* idx,
                        double* score_out)
{
    if (B <= 0 || N <= 0 || C <= 0 || K < 0 || K > N) return 1;
    double* mean = (double*)malloc(sizeof(double) * (size_t)B * C);
    double* score = (double*)malloc(sizeof(double) * (size_t)B * N);
    scored* order = (scored*)malloc(sizeof(scored) * (size_t)N);
    if (!mean || !score || !order) { free(mean); free(score); free(order); return 2; }
    oracle_pivot_mean(B, N, C, x, mean);
    oracle_pivot_scores(B, N, C, x, mean, score);
    for (int b = 0; b < B; b++) {
        for (int i = 0; i < N; i++) { order[i].s = score[(size_t)b * N + i]; order[i].i = i; }
        qsort(order, (size_t)N, sizeof(scored), by_score_desc);
        for (int j = 0; j < K; j++) idx[(size_t)b * K + j] = order[j].i;
        qsort(idx + (size_t)b * K, (size_t)K, sizeof(int32_t), by_int_asc);
    }
    if (score_out) memcpy(score_out, score, sizeof(double) * (size_t)B * N);
    free(mean); free(score); free(order);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Structural reconstruction: Up(prev) then overwrite kept rows         */
/* ------------------------------------------------------------------ */

/* Source coordinate of output pixel dst for an in->out resize (half-pixel centres). */
static void bilinear_axis(int dst, int in, int out, int* i0, int* i1, double* lam)
{
    double src = ((double)dst + 0.5) * (double)in / (double)out - 0.5;
    if (src < 0.0) src = 0.0;
    int a = (int)floor(src);
    if (a > in - 1) a = in - 1;
    *i0 = a;
    *i1 = (a < in - 1) ? a + 1 : a;
    *lam = src - (double)a;
}

/*
 * out[b][h][n][:] = bilinear upsample of prev ([B][H][sp*sp][D], grid sp x sp)
 * to the s x s grid, then out[b][h][idx[b][j]][:] = oc[b][h][j][:] for j < K.
 * idx must be strictly ascending and inside [0, s*s).
 */
int oracle_restore_scatter(int B, int H, int sp, int s, int D, const uint16_t* prev,
                           const uint16_t* oc, const int32_t* idx, int K, double* out)
{
    if (B <= 0 || H <= 0 || sp <= 0 || s <= 0 || D <= 0 || K < 0 || K > s * s) return 1;
    for (int b = 0; b < B; b++)
        for (int j = 0; j < K; j++) {
            const int32_t n = idx[(size_t)b * K + j];
            if (n < 0 || n >= s * s) return 1;
            if (j > 0 && n <= idx[(size_t)b * K + j - 1]) return 1;
        }
    const int N = s * s, Np = sp * sp;
#pragma omp parallel for schedule(static)
    for (long bh = 0; bh < (long)B * H; bh++) {
        const uint16_t* P = prev + (size_t)bh * Np * D;
        double* O = out + (size_t)bh * N * D;
        for (int y = 0; y < s; y++) {
            int y0, y1; double ly;
            bilinear_axis(y, sp, s, &y0, &y1, &ly);
            for (int x = 0; x < s; x++) {
                int x0, x1; double lx;
                bilinear_axis(x, sp, s, &x0, &x1, &lx);
                for (int d = 0; d < D; d++) {
                    const double a00 = bf16_to_f64(P[((size_t)y0 * sp + x0) * D + d]);
                    const double a01 = bf16_to_f64(P[((size_t)y0 * sp + x1) * D + d]);
                    const double a10 = bf16_to_f64(P[((size_t)y1 * sp + x0) * D + d]);
                    const double a11 = bf16_to_f64(P[((size_t)y1 * sp + x1) * D + d]);
                    const double top = (1.0 - lx) * a00 + lx * a01;
                    const double bot = (1.0 - lx) * a10 + lx * a11;
                    O[((size_t)y * s + x) * D + d] = (1.0 - ly) * top + ly * bot;
                }
            }
        }
        const long b = bh / H;
        for (int j = 0; j < K; j++) {
            const int n = idx[(size_t)b * K + j];
            for (int d = 0; d < D; d++)
                O[(size_t)n * D + d] = bf16_to_f64(oc[((size_t)bh * K + j) * D + d]);
        }
    }
    return 0;
}

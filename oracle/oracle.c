/*
 * oracle.c -- plain, slow, fp64 CPU definition of FlashMask masked attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  The CUDA library never
 * does, and this file shares no code, header or constant with it.
 *
 * What is computed, and where it is defined:
 *
 *  - FlashMask README (PaddlePaddle/FlashMask), "Formulation":
 *        O = softmax(Q K^T / sqrt(d) + M) V
 *    d is the last dimension of Q (the Q/K head dim).  M is additive: 0 where
 *    the pair (i, j) is visible and -inf where it is masked.  The caller passes
 *    the softmax scale, 1/sqrt(d) by default.
 *
 *  - FlashMask README, "Overview", and "FlashMask-3: Efficient and Expressive
 *    Mask-Aware Distributed Attention", abstract: the mask is stored
 *    column-wise.  Key column j holds four query-axis boundaries.  Row i is
 *    masked in column j when LTS_j <= i < LTE_j or UTS_j <= i < UTE_j.  A
 *    causal flag additionally masks every i < j.  A NULL boundary pair means
 *    that interval is empty.
 *
 *  - Rows with every key masked: O = 0 and LSE = -inf.  The row contributes
 *    nothing to dQ, dK or dV.  The pages do not fix this case; this is the
 *    stated convention.
 *
 *  - Backward: the textbook derivative of the formula above.  With P the
 *    softmax probabilities, dP = dO V^T, D_i = sum_j P_ij dP_ij and
 *    dS = P * (dP - D):  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 *
 *  - Tile map: a (q-tile, k-tile) block is SKIP when every in-range element is
 *    masked, UNMASKED when none is, else PARTIAL.  This is the brute-force count
 *    behind the sparsity skipping of "FlashMask: Efficient and Rich Mask
 *    Extension of FlashAttention", abstract.
 *
 * Everything is computed in double precision from the exact input values.
 * Rows are independent, so OpenMP runs them in parallel; nothing is blocked,
 * fused or reordered beyond that.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Tile classes of the tile map. */
#define ORACLE_TILE_SKIP 0
#define ORACLE_TILE_PARTIAL 1
#define ORACLE_TILE_UNMASKED 2

typedef struct {
    int N;
    int causal;
    const int32_t *lts, *lte, *uts, *ute;
} oracle_mask;

/* The column-wise sparse mask predicate: 1 when row i may not see key j. */
static int oracle_is_masked(const oracle_mask *m, long i, long j)
{
    if (m->causal && i < j)
        return 1;
    if (m->lts && m->lte && m->lts[j] <= i && i < m->lte[j])
        return 1;
    if (m->uts && m->ute && m->uts[j] <= i && i < m->ute[j])
        return 1;
    return 0;
}

static double oracle_dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int c = 0; c < n; ++c)
        s += a[c] * b[c];
    return s;
}

/* Scores of query row i: s_j = scale * <q_i, k_j>, or -inf where masked.
 * Returns max_j s_j (-inf when the whole row is masked). */
static double oracle_row_scores(const oracle_mask *m, int d, double scale,
                                const double *q, const double *k, long i,
                                double *s)
{
    double mx = -INFINITY;
    for (long j = 0; j < m->N; ++j) {
        if (oracle_is_masked(m, i, j)) {
            s[j] = -INFINITY;
        } else {
            s[j] = scale * oracle_dot(q + i * d, k + j * d, d);
            if (s[j] > mx)
                mx = s[j];
        }
    }
    return mx;
}

/* Softmax of one row in place: s_j <- P_ij.  Returns LSE_i = log(exp(sink) +
 * sum_j exp(s_j)).  `sink` is the row's attention-sink logit, a term of the
 * denominator that carries no value (-inf: none); *p_sink (optional) receives
 * its probability exp(sink - LSE_i).  A row with every key masked and no sink
 * gives P = 0 and LSE = -inf. */
static double oracle_row_softmax(long N, double mx, double sink, double *s, double *p_sink)
{
    if (sink > mx)
        mx = sink;
    if (mx == -INFINITY) {
        for (long j = 0; j < N; ++j)
            s[j] = 0.0;
        if (p_sink)
            *p_sink = 0.0;
        return -INFINITY;
    }
    double l = (sink == -INFINITY) ? 0.0 : exp(sink - mx);
    for (long j = 0; j < N; ++j) {
        s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - mx);
        l += s[j];
    }
    for (long j = 0; j < N; ++j)
        s[j] /= l;
    if (p_sink)
        *p_sink = (sink == -INFINITY) ? 0.0 : exp(sink - mx) / l;
    return mx + log(l);
}

/*
 * Forward for one (batch, head) slice.
 *   q, k: [N, d]; v: [N, dv] (row-major, fp64 copies of the inputs)
 *   rows: n_rows query indices, or NULL for all N rows
 *   o: [n_rows, dv]; lse: [n_rows] (natural log)
 */
int oracle_fwd(int N, int d, int dv, double scale, int causal, double sink,
               const double *q, const double *k, const double *v,
               const int32_t *lts, const int32_t *lte,
               const int32_t *uts, const int32_t *ute,
               long n_rows, const int64_t *rows, double *o, double *lse)
{
    oracle_mask m = {N, causal, lts, lte, uts, ute};
    if (!rows)
        n_rows = N;
    int err = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)N);
        if (!p) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < n_rows; ++r) {
            if (!p)
                continue;
            long i = rows ? (long)rows[r] : r;
            double mx = oracle_row_scores(&m, d, scale, q, k, i, p);
            lse[r] = oracle_row_softmax(N, mx, sink, p, NULL);
            for (int c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (long j = 0; j < N; ++j)
                    if (p[j] != 0.0)
                        acc += p[j] * v[j * dv + c];
                o[r * dv + c] = acc;
            }
        }
        free(p);
    }
    return err;
}

/*
 * Backward, query side, for selected rows of one (batch, head) slice.
 *   dout: [N, dv];  dq: [n_rows, d];  delta (optional): [n_rows], D_i;
 *   dsink (optional): [n_rows], the row's term of the sink logit's gradient.
 * dQ_i = scale * sum_j P_ij (dP_ij - D_i) k_j, dP_ij = <dO_i, v_j>.  The sink
 * carries no value, so its dP is 0 and its gradient term is -P_sink,i D_i.
 */
int oracle_bwd_dq(int N, int d, int dv, double scale, int causal, double sink,
                  const double *q, const double *k, const double *v,
                  const double *dout,
                  const int32_t *lts, const int32_t *lte,
                  const int32_t *uts, const int32_t *ute,
                  long n_rows, const int64_t *rows, double *dq, double *delta,
                  double *dsink)
{
    oracle_mask m = {N, causal, lts, lte, uts, ute};
    if (!rows)
        n_rows = N;
    int err = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)N);
        double *dp = (double *)malloc(sizeof(double) * (size_t)N);
        if (!p || !dp) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < n_rows; ++r) {
            if (!p || !dp)
                continue;
            long i = rows ? (long)rows[r] : r;
            double mx = oracle_row_scores(&m, d, scale, q, k, i, p);
            double p_sink = 0.0;
            oracle_row_softmax(N, mx, sink, p, &p_sink);
            double D = 0.0;
            for (long j = 0; j < N; ++j) {
                dp[j] = (p[j] != 0.0) ? oracle_dot(dout + i * dv, v + j * dv, dv) : 0.0;
                D += p[j] * dp[j];
            }
            if (delta)
                delta[r] = D;
            if (dsink)
                dsink[r] = -p_sink * D;
            for (int c = 0; c < d; ++c)
                dq[r * d + c] = 0.0;
            for (long j = 0; j < N; ++j) {
                if (p[j] == 0.0)
                    continue;
                double ds = p[j] * (dp[j] - D);
                for (int c = 0; c < d; ++c)
                    dq[r * d + c] += scale * ds * k[j * d + c];
            }
        }
        free(p);
        free(dp);
    }
    return err;
}

/*
 * Backward, key side, for selected key columns of one (batch, head) slice.
 *   cols: n_cols key indices, or NULL for all N columns
 *   dk: [n_cols, d]; dvv: [n_cols, dv]
 * dK_j = scale * sum_i P_ij (dP_ij - D_i) q_i,  dV_j = sum_i P_ij dO_i.
 * Every row that sees one of the columns first gets its LSE_i and D_i from a
 * full pass over that row; the columns are then summed over rows in order.
 */
int oracle_bwd_dkdv(int N, int d, int dv, double scale, int causal, double sink,
                    const double *q, const double *k, const double *v,
                    const double *dout,
                    const int32_t *lts, const int32_t *lte,
                    const int32_t *uts, const int32_t *ute,
                    long n_cols, const int64_t *cols, double *dk, double *dvv)
{
    oracle_mask m = {N, causal, lts, lte, uts, ute};
    if (!cols)
        n_cols = N;
    double *row_lse = (double *)malloc(sizeof(double) * (size_t)N);
    double *row_D = (double *)malloc(sizeof(double) * (size_t)N);
    unsigned char *need = (unsigned char *)calloc((size_t)N, 1);
    if (!row_lse || !row_D || !need) {
        free(row_lse);
        free(row_D);
        free(need);
        return 1;
    }
    /* Which rows see at least one requested column. */
#pragma omp parallel for schedule(dynamic, 64)
    for (long i = 0; i < N; ++i) {
        for (long c = 0; c < n_cols; ++c) {
            long j = cols ? (long)cols[c] : c;
            if (!oracle_is_masked(&m, i, j)) {
                need[i] = 1;
                break;
            }
        }
    }
    int err = 0;
    /* Row statistics LSE_i and D_i for those rows. */
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)N);
        if (!p) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long i = 0; i < N; ++i) {
            if (!p || !need[i])
                continue;
            double mx = oracle_row_scores(&m, d, scale, q, k, i, p);
            row_lse[i] = oracle_row_softmax(N, mx, sink, p, NULL);
            double D = 0.0;
            for (long j = 0; j < N; ++j)
                if (p[j] != 0.0)
                    D += p[j] * oracle_dot(dout + i * dv, v + j * dv, dv);
            row_D[i] = D;
        }
        free(p);
    }
    /* Column sums. */
#pragma omp parallel for schedule(dynamic, 1)
    for (long c = 0; c < n_cols; ++c) {
        long j = cols ? (long)cols[c] : c;
        double *dkj = dk + c * d;
        double *dvj = dvv + c * dv;
        for (int x = 0; x < d; ++x)
            dkj[x] = 0.0;
        for (int x = 0; x < dv; ++x)
            dvj[x] = 0.0;
        for (long i = 0; i < N; ++i) {
            if (oracle_is_masked(&m, i, j) || row_lse[i] == -INFINITY)
                continue;
            double s = scale * oracle_dot(q + i * d, k + j * d, d);
            double pij = exp(s - row_lse[i]);
            double dpij = oracle_dot(dout + i * dv, v + j * dv, dv);
            double ds = pij * (dpij - row_D[i]);
            for (int x = 0; x < d; ++x)
                dkj[x] += scale * ds * q[i * d + x];
            for (int x = 0; x < dv; ++x)
                dvj[x] += pij * dout[i * dv + x];
        }
    }
    free(row_lse);
    free(row_D);
    free(need);
    return err;
}

/*
 * Brute-force tile map: tq x tk tiles aligned to 0; a tile at the ragged edge
 * counts only the in-range elements.  cls: [ceil(N/tq), ceil(N/tk)].
 * Returns the number of unmasked (i, j) pairs over the whole N x N square.
 */
long long oracle_tilemap(int N, int causal,
                         const int32_t *lts, const int32_t *lte,
                         const int32_t *uts, const int32_t *ute,
                         int tq, int tk, int8_t *cls)
{
    oracle_mask m = {N, causal, lts, lte, uts, ute};
    long nq = (N + tq - 1) / tq, nk = (N + tk - 1) / tk;
    long long total_visible = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : total_visible)
    for (long t = 0; t < nq * nk; ++t) {
        long qt = t / nk, kt = t % nk;
        long i1 = (qt + 1) * tq < N ? (qt + 1) * tq : N;
        long j1 = (kt + 1) * tk < N ? (kt + 1) * tk : N;
        long n_in = 0, n_masked = 0;
        for (long i = qt * tq; i < i1; ++i)
            for (long j = kt * tk; j < j1; ++j) {
                ++n_in;
                n_masked += oracle_is_masked(&m, i, j);
            }
        if (cls)
            cls[t] = (n_masked == n_in) ? ORACLE_TILE_SKIP
                     : (n_masked == 0) ? ORACLE_TILE_UNMASKED
                                       : ORACLE_TILE_PARTIAL;
        total_visible += n_in - n_masked;
    }
    return total_visible;
}

/* Number of threads OpenMP runs with (for reporting). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * CPU oracle for the backward pass of exact softmax attention — TEST
 * INFRASTRUCTURE ONLY (same rules as attn_oracle.c: only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load it).
 *
 * What it computes, in fp64, for upstream gradient dO of the output:
 *
 *   S = scale * Q K^T,  P = softmax(S) row-wise,  O = P V
 *   dV = P^T dO
 *   dP = dO V^T
 *   dS_ij = P_ij * (dP_ij - D_i),   D_i = sum_j P_ij dP_ij
 *   dQ = scale * dS K,   dK = scale * dS^T Q
 *
 * The pages say only that the backward pass recomputes the attention blocks
 * from Q, K, V and the saved softmax statistics instead of storing the N x N
 * matrix ("FlashAttention dissected", section "Memory complexity: from O(N^2)
 * to O(N)").  They give no gradient formulas, so the oracle takes the plain
 * reading: the exact gradient of the forward definition (the softmax formula
 * of the same page's section "The mathematical breakthrough: Tiling and
 * Online Softmax", whose Jacobian is dP_j/dS_k = P_j (delta_jk - P_k)),
 * obtained by the chain rule through O = P V and S = scale Q K^T.
 *
 * Each query row is evaluated on its own, like the forward oracle: its scores
 * in an fp64 buffer, the softmax by three passes (maximum, sum of shifted
 * exponentials, normalised weights), then dP, D and dS for that row; dQ is
 * that row's, and the row's contributions are added into dK and dV of its
 * key/value head.  Nothing here uses the saved lse: P is recomputed from
 * its definition.
 *
 * Shapes and conventions are those of attn_oracle.c: q, dO fp32
 * [B, H, Nq, d]; k, v fp32 [B, H_kv, Nkv, d], query head h uses key/value
 * head h / (H / H_kv); causal: query i sees keys j <= i + (Nkv - Nq).  A row
 * with no visible key has P = 0 and contributes nothing.
 *
 * Parity is pinned by tests/test_oracle_bwd_pins.py (finite differences of
 * the forward oracle, automatic differentiation in fp64, closed forms and
 * invariants).  ORACLE_MUTANT values 11-16 plant mistakes for those tests.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

typedef struct {
    const float *q, *k, *v, *dout;
    int64_t B, H, H_kv, Nq, Nkv, d;
    int causal;
    double scale;
} problem_t;

/* keys visible to query row i: all Nkv, or the causal prefix (may be 0) */
static int64_t visible_keys(const problem_t *pb, int64_t i)
{
    int64_t n = pb->Nkv;
#if ORACLE_MUTANT == 15 /* causal mask forgotten in the backward pass */
    (void)i;
#else
    if (pb->causal && i + (pb->Nkv - pb->Nq) + 1 < n)
        n = i + (pb->Nkv - pb->Nq) + 1;
#endif
    return n < 0 ? 0 : n;
}

/*
 * One query row (b, h, i): fills p[0..n) with the softmax weights,
 * dp[0..n) with dO_i . v_j, and returns n, the visible key count; *D gets
 * sum_j p_j dp_j.  s is scratch of Nkv doubles.
 */
static int64_t row_terms(const problem_t *pb, int64_t b, int64_t h, int64_t i,
                         double *s, double *p, double *dp, double *D)
{
    const int64_t d = pb->d;
    const int64_t kvh = b * pb->H_kv + h / (pb->H / pb->H_kv);
    const float *q_row = pb->q + ((b * pb->H + h) * pb->Nq + i) * d;
    const float *do_row = pb->dout + ((b * pb->H + h) * pb->Nq + i) * d;
    const float *kh = pb->k + kvh * pb->Nkv * d;
    const float *vh = pb->v + kvh * pb->Nkv * d;
    const int64_t n = visible_keys(pb, i);
    int64_t j, c;

    *D = 0.0;
    if (n == 0)
        return 0;
    for (j = 0; j < n; ++j) {
        double acc = 0.0;
        for (c = 0; c < d; ++c)
            acc += (double)q_row[c] * (double)kh[j * d + c];
        s[j] = pb->scale * acc;
    }
    /* softmax: maximum, sum of shifted exponentials, normalised weights */
    double m = -INFINITY;
    for (j = 0; j < n; ++j)
        if (s[j] > m)
            m = s[j];
    double l = 0.0;
    for (j = 0; j < n; ++j)
        l += exp(s[j] - m);
    for (j = 0; j < n; ++j)
        p[j] = exp(s[j] - m) / l;
    /* dP_ij = dO_i . v_j and D_i = sum_j P_ij dP_ij */
    double acc_D = 0.0;
    for (j = 0; j < n; ++j) {
        double acc = 0.0;
        for (c = 0; c < d; ++c)
            acc += (double)do_row[c] * (double)vh[j * d + c];
        dp[j] = acc;
        acc_D += p[j] * dp[j];
    }
    *D = acc_D;
    return n;
}

/* dS_ij = P_ij (dP_ij - D_i) */
static double grad_score(double p, double dp, double D)
{
#if ORACLE_MUTANT == 11 /* the -D_i term dropped */
    (void)D;
    return p * dp;
#else
    return p * (dp - D);
#endif
}

/*
 * Every gradient of one (batch b, key/value head kvh) unit: the query rows
 * of its H / H_kv query heads add into dk, dv of that key/value head, and
 * each row's dq is written.  dq: fp64 [B, H, Nq, d]; dk, dv: fp64
 * [B, H_kv, Nkv, d] (the unit's slices are zeroed here first).
 */
static int unit_backward(const problem_t *pb, int64_t b, int64_t kvh,
                         double *dq, double *dk, double *dv)
{
    const int64_t d = pb->d, Nkv = pb->Nkv, group = pb->H / pb->H_kv;
    const size_t n_buf = (size_t)(Nkv > 0 ? Nkv : 1);
    double *s = (double *)malloc(n_buf * sizeof(double));
    double *p = (double *)malloc(n_buf * sizeof(double));
    double *dp = (double *)malloc(n_buf * sizeof(double));
    if (!s || !p || !dp) {
        free(s); free(p); free(dp);
        return -2;
    }
    const int64_t unit = b * pb->H_kv + kvh;
    double *dk_h = dk + unit * Nkv * d;
    double *dv_h = dv + unit * Nkv * d;
    const float *kh = pb->k + unit * Nkv * d;
    memset(dk_h, 0, (size_t)(Nkv * d) * sizeof(double));
    memset(dv_h, 0, (size_t)(Nkv * d) * sizeof(double));

    for (int64_t g = 0; g < group; ++g) {
        const int64_t h = kvh * group + g;
        for (int64_t i = 0; i < pb->Nq; ++i) {
            const int64_t row = (b * pb->H + h) * pb->Nq + i;
            const float *q_row = pb->q + row * d;
            const float *do_row = pb->dout + row * d;
            double *dq_row = dq + row * d;
            double D;
            const int64_t n = row_terms(pb, b, h, i, s, p, dp, &D);
            for (int64_t c = 0; c < d; ++c)
                dq_row[c] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                const double ds = grad_score(p[j], dp[j], D);
                for (int64_t c = 0; c < d; ++c) {
#if ORACLE_MUTANT == 14 /* transposed K operand in dQ */
                    dq_row[c] += ds * (double)kh[c * Nkv + j];
#else
                    dq_row[c] += ds * (double)kh[j * d + c];
#endif
#if ORACLE_MUTANT == 12 /* dK without the score scale */
                    dk_h[j * d + c] += ds * (double)q_row[c];
#else
                    dk_h[j * d + c] += pb->scale * ds * (double)q_row[c];
#endif
#if ORACLE_MUTANT == 13 /* dV weighted by dP instead of P */
                    dv_h[j * d + c] += dp[j] * (double)do_row[c];
#else
                    dv_h[j * d + c] += p[j] * (double)do_row[c];
#endif
                }
            }
            for (int64_t c = 0; c < d; ++c)
#if ORACLE_MUTANT == 16 /* dQ without the score scale */
                dq_row[c] = dq_row[c];
#else
                dq_row[c] *= pb->scale;
#endif
        }
    }
    free(s); free(p); free(dp);
    return 0;
}

typedef struct {
    const problem_t *pb;
    double *dq, *dk, *dv;
    int64_t first, last; /* half-open range of units (b * H_kv + kvh) */
    int status;
} bwd_job_t;

static void *bwd_worker(void *arg)
{
    bwd_job_t *jb = (bwd_job_t *)arg;
    for (int64_t u = jb->first; u < jb->last && jb->status == 0; ++u)
        jb->status = unit_backward(jb->pb, u / jb->pb->H_kv, u % jb->pb->H_kv,
                                   jb->dq, jb->dk, jb->dv);
    return NULL;
}

int oracle_default_threads(void);

/* Run fn on jobs[0..threads) (job_size bytes apart), one thread each; jobs
   whose thread could not be started run on this one. */
typedef void *(*job_fn)(void *);
static int run_jobs(job_fn fn, void *jobs, size_t job_size, int threads)
{
    pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    if (!tids)
        return -2;
    int launched = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tids[t], NULL, fn, (char *)jobs + (size_t)t * job_size) != 0)
            break;
        launched = t;
    }
    fn(jobs);
    for (int t = launched + 1; t < threads; ++t)
        fn((char *)jobs + (size_t)t * job_size);
    for (int t = 1; t <= launched; ++t)
        pthread_join(tids[t], NULL);
    free(tids);
    return 0;
}

static int check_problem(const problem_t *pb)
{
    if (!pb->q || !pb->k || !pb->v || !pb->dout || pb->B < 1 || pb->H < 1 || pb->H_kv < 1 ||
        pb->H % pb->H_kv != 0 || pb->Nq < 1 || pb->Nkv < 1 || pb->d < 1)
        return -1;
    return 0;
}

/*
 * Gradients of exact attention, every element, in fp64.
 *   q, dout : fp32 [B, H, Nq, d];  k, v : fp32 [B, H_kv, Nkv, d]
 *   dq      : fp64 [B, H, Nq, d];  dk, dv : fp64 [B, H_kv, Nkv, d]
 *   threads : worker count, 0 = every online core (work is split by
 *             (b, key/value head) unit).
 * Returns 0, -1 on a bad argument, -2 when memory runs out.
 */
int oracle_attention_bwd_f64(const float *q, const float *k, const float *v,
                             const float *dout, int64_t B, int64_t H, int64_t H_kv,
                             int64_t Nq, int64_t Nkv, int64_t d, double scale,
                             int causal, double *dq, double *dk, double *dv,
                             int threads)
{
    problem_t pb = {q, k, v, dout, B, H, H_kv, Nq, Nkv, d, causal, scale};
    if (check_problem(&pb) != 0 || !dq || !dk || !dv)
        return -1;
    const int64_t units = B * H_kv;
    if (threads <= 0)
        threads = oracle_default_threads();
    if ((int64_t)threads > units)
        threads = (int)units;
    bwd_job_t *jobs = (bwd_job_t *)calloc((size_t)threads, sizeof(bwd_job_t));
    if (!jobs)
        return -2;
    for (int t = 0; t < threads; ++t) {
        jobs[t].pb = &pb;
        jobs[t].dq = dq; jobs[t].dk = dk; jobs[t].dv = dv;
        jobs[t].first = units * t / threads;
        jobs[t].last = units * (t + 1) / threads;
    }
    int status = run_jobs(bwd_worker, jobs, sizeof(bwd_job_t), threads);
    for (int t = 0; t < threads && status == 0; ++t)
        status = jobs[t].status;
    free(jobs);
    return status;
}

/* ------------------------------------------------------------------------
 * Sampled gradients for large problems.  dQ of a row depends on that row
 * alone; dK and dV of a key need every query row of its key/value head.
 * ---------------------------------------------------------------------- */

typedef struct {
    const problem_t *pb;
    const int64_t *rows; /* (b, h, i) triples */
    double *dq;          /* [nrows, d] */
    int64_t first, last;
    int status;
} dq_job_t;

static void *dq_worker(void *arg)
{
    dq_job_t *jb = (dq_job_t *)arg;
    const problem_t *pb = jb->pb;
    const int64_t d = pb->d;
    const size_t n_buf = (size_t)pb->Nkv;
    double *s = (double *)malloc(n_buf * sizeof(double));
    double *p = (double *)malloc(n_buf * sizeof(double));
    double *dp = (double *)malloc(n_buf * sizeof(double));
    if (!s || !p || !dp) {
        free(s); free(p); free(dp);
        jb->status = -2;
        return NULL;
    }
    for (int64_t r = jb->first; r < jb->last; ++r) {
        const int64_t b = jb->rows[3 * r], h = jb->rows[3 * r + 1], i = jb->rows[3 * r + 2];
        const int64_t kvh = b * pb->H_kv + h / (pb->H / pb->H_kv);
        const float *kh = pb->k + kvh * pb->Nkv * d;
        double *dq_row = jb->dq + r * d;
        double D;
        const int64_t n = row_terms(pb, b, h, i, s, p, dp, &D);
        for (int64_t c = 0; c < d; ++c)
            dq_row[c] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            const double ds = grad_score(p[j], dp[j], D);
            for (int64_t c = 0; c < d; ++c)
                dq_row[c] += ds * (double)kh[j * d + c];
        }
        for (int64_t c = 0; c < d; ++c)
            dq_row[c] *= pb->scale;
    }
    free(s); free(p); free(dp);
    return NULL;
}

/*
 * dQ rows (b, h, i) of `rows` (nrows triples) into dq fp64 [nrows, d].
 * Returns 0, -1 on a bad argument or out-of-range triple, -2 on memory.
 */
int oracle_attention_bwd_dq_rows_f64(const float *q, const float *k, const float *v,
                                     const float *dout, int64_t B, int64_t H, int64_t H_kv,
                                     int64_t Nq, int64_t Nkv, int64_t d, double scale,
                                     int causal, const int64_t *rows, int64_t nrows,
                                     double *dq, int threads)
{
    problem_t pb = {q, k, v, dout, B, H, H_kv, Nq, Nkv, d, causal, scale};
    if (check_problem(&pb) != 0 || !rows || !dq || nrows < 0)
        return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t *t = rows + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= H || t[2] < 0 || t[2] >= Nq)
            return -1;
    }
    if (nrows == 0)
        return 0;
    if (threads <= 0)
        threads = oracle_default_threads();
    if ((int64_t)threads > nrows)
        threads = (int)nrows;
    dq_job_t *jobs = (dq_job_t *)calloc((size_t)threads, sizeof(dq_job_t));
    if (!jobs)
        return -2;
    for (int t = 0; t < threads; ++t) {
        jobs[t].pb = &pb;
        jobs[t].rows = rows;
        jobs[t].dq = dq;
        jobs[t].first = nrows * t / threads;
        jobs[t].last = nrows * (t + 1) / threads;
    }
    int status = run_jobs(dq_worker, jobs, sizeof(dq_job_t), threads);
    for (int t = 0; t < threads && status == 0; ++t)
        status = jobs[t].status;
    free(jobs);
    return status;
}

typedef struct {
    const problem_t *pb;
    int64_t b, kvh;        /* the unit */
    const int64_t *keys;   /* key indices j requested in this unit */
    int64_t nkeys;
    int64_t first, last;   /* half-open range of the unit's query rows g * Nq + i */
    double *dk, *dv;       /* this worker's partial sums [nkeys, d] */
    int status;
} dkv_job_t;

static void *dkv_worker(void *arg)
{
    dkv_job_t *jb = (dkv_job_t *)arg;
    const problem_t *pb = jb->pb;
    const int64_t d = pb->d, group = pb->H / pb->H_kv;
    const size_t n_buf = (size_t)pb->Nkv;
    double *s = (double *)malloc(n_buf * sizeof(double));
    double *p = (double *)malloc(n_buf * sizeof(double));
    double *dp = (double *)malloc(n_buf * sizeof(double));
    if (!s || !p || !dp) {
        free(s); free(p); free(dp);
        jb->status = -2;
        return NULL;
    }
    for (int64_t r = jb->first; r < jb->last; ++r) {
        const int64_t h = jb->kvh * group + r / pb->Nq, i = r % pb->Nq;
        const int64_t row = (jb->b * pb->H + h) * pb->Nq + i;
        const float *q_row = pb->q + row * d;
        const float *do_row = pb->dout + row * d;
        double D;
        const int64_t n = row_terms(pb, jb->b, h, i, s, p, dp, &D);
        for (int64_t c = 0; c < jb->nkeys; ++c) {
            const int64_t j = jb->keys[c];
            if (j >= n)
                continue; /* key not visible to this row */
            const double ds = grad_score(p[j], dp[j], D);
            for (int64_t e = 0; e < d; ++e) {
                jb->dk[c * d + e] += pb->scale * ds * (double)q_row[e];
                jb->dv[c * d + e] += p[j] * (double)do_row[e];
            }
        }
    }
    free(s); free(p); free(dp);
    return NULL;
}

/*
 * dK and dV of the keys (b, kvh, j) in `cols` (ncols triples) into dk, dv
 * fp64 [ncols, d].  Keys are grouped by (b, kvh) unit; for each unit every
 * query row of its query heads is evaluated once (threads split the rows,
 * their partial sums are added in thread order).
 * Returns 0, -1 on a bad argument or out-of-range triple, -2 on memory.
 */
int oracle_attention_bwd_dkv_cols_f64(const float *q, const float *k, const float *v,
                                      const float *dout, int64_t B, int64_t H, int64_t H_kv,
                                      int64_t Nq, int64_t Nkv, int64_t d, double scale,
                                      int causal, const int64_t *cols, int64_t ncols,
                                      double *dk, double *dv, int threads)
{
    problem_t pb = {q, k, v, dout, B, H, H_kv, Nq, Nkv, d, causal, scale};
    if (check_problem(&pb) != 0 || !cols || !dk || !dv || ncols < 0)
        return -1;
    for (int64_t c = 0; c < ncols; ++c) {
        const int64_t *t = cols + 3 * c;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= H_kv || t[2] < 0 || t[2] >= Nkv)
            return -1;
    }
    memset(dk, 0, (size_t)(ncols * d) * sizeof(double));
    memset(dv, 0, (size_t)(ncols * d) * sizeof(double));
    if (ncols == 0)
        return 0;
    const int64_t rows_per_unit = (H / H_kv) * Nq;
    if (threads <= 0)
        threads = oracle_default_threads();
    if ((int64_t)threads > rows_per_unit)
        threads = (int)rows_per_unit;

    int64_t *keys = (int64_t *)malloc((size_t)ncols * sizeof(int64_t));
    int64_t *slot = (int64_t *)malloc((size_t)ncols * sizeof(int64_t));
    char *done = (char *)calloc((size_t)ncols, 1);
    dkv_job_t *jobs = (dkv_job_t *)calloc((size_t)threads, sizeof(dkv_job_t));
    double *part = (double *)malloc((size_t)threads * 2 * (size_t)(ncols * d) * sizeof(double));
    int status = 0;
    if (!keys || !slot || !done || !jobs || !part)
        status = -2;
    for (int64_t c0 = 0; c0 < ncols && status == 0; ++c0) {
        if (done[c0])
            continue;
        /* every requested key of the unit of cols[c0] */
        const int64_t b = cols[3 * c0], kvh = cols[3 * c0 + 1];
        int64_t nk = 0;
        for (int64_t c = c0; c < ncols; ++c) {
            if (!done[c] && cols[3 * c] == b && cols[3 * c + 1] == kvh) {
                keys[nk] = cols[3 * c + 2];
                slot[nk] = c;
                done[c] = 1;
                ++nk;
            }
        }
        memset(part, 0, (size_t)threads * 2 * (size_t)(nk * d) * sizeof(double));
        for (int t = 0; t < threads; ++t) {
            dkv_job_t *jb = &jobs[t];
            jb->pb = &pb;
            jb->b = b;
            jb->kvh = kvh;
            jb->keys = keys;
            jb->nkeys = nk;
            jb->first = rows_per_unit * t / threads;
            jb->last = rows_per_unit * (t + 1) / threads;
            jb->dk = part + (size_t)(2 * t) * (size_t)(nk * d);
            jb->dv = part + (size_t)(2 * t + 1) * (size_t)(nk * d);
            jb->status = 0;
        }
        status = run_jobs(dkv_worker, jobs, sizeof(dkv_job_t), threads);
        for (int t = 0; t < threads && status == 0; ++t) {
            status = jobs[t].status;
            for (int64_t c = 0; c < nk; ++c)
                for (int64_t e = 0; e < d; ++e) {
                    dk[slot[c] * d + e] += jobs[t].dk[c * d + e];
                    dv[slot[c] * d + e] += jobs[t].dv[c * d + e];
                }
        }
    }
    free(keys); free(slot); free(done); free(jobs); free(part);
    return status;
}

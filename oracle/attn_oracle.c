/*
 * CPU oracle for exact softmax attention — TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  The GPU product path never calls it.
 *
 * What it computes (the plain definition, in fp64):
 *
 *   O = softmax(scale * Q K^T) V          per (batch b, head h)
 *   lse_i = log( sum_j exp(scale * q_i . k_j) )        natural log
 *
 *   - "CUDA Flash Attention: Online Softmax with Shared Memory Tiling",
 *     Problem Statement: attention is softmax(Q K^T / sqrt(d)) V; here the
 *     1/sqrt(d) factor is the caller's `scale` (the same page's fused kernel
 *     takes `scale` as an argument).
 *   - "FlashAttention dissected", section "The mathematical breakthrough:
 *     Tiling and Online Softmax": softmax(x)_i = e^{x_i} / sum_j e^{x_j}.
 *   - "How Did I Write My First FlashAttention Kernel in CUDA?", the
 *     paragraph on the three passes a plain softmax needs: (1) the row
 *     maximum, (2) the sum of exponentials shifted by that maximum,
 *     (3) the normalised weights.  Pass 3 is fused with the weighted sum
 *     of V rows, which is still a plain evaluation of the definition.
 *   - lse (log-sum-exp) is the per-row statistic "FlashAttention dissected",
 *     section "Memory complexity: from O(N^2) to O(N)", says is kept for
 *     the backward pass (the maximum m and the denominator l); it is
 *     reported as the single number m + ln(l).
 *
 * No tiling, no online rescaling, no reordering: one query row at a time,
 * all N scores of that row held in an fp64 buffer, three passes over it.
 *
 * Inputs are fp32 arrays holding values already rounded to the kernel's
 * input dtype (bf16 values are exactly representable in fp32); every value
 * is widened to double before use.  Layout: contiguous row-major
 * [B, H, N, d].
 *
 * Parity is pinned by tests/test_oracle_pins.py (closed forms, invariants,
 * a library routine and brute force on tiny inputs).
 *
 * ORACLE_MUTANT (compile-time, default 0) plants a deliberate mistake so the
 * test suite can prove that its pins catch it.  Products are built with 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* One query row: o_row[0..d) and *lse from q_row, the head's K and V. */
static void attention_row(const float *q_row, const float *k_head,
                          const float *v_head, int64_t N, int64_t d,
                          double scale, double *s, double *o_row,
                          double *lse)
{
    int64_t j, c;

    /* scores s_j = scale * sum_c q[c] k[j, c] */
    for (j = 0; j < N; ++j) {
        double acc = 0.0;
        for (c = 0; c < d; ++c) {
#if ORACLE_MUTANT == 2 /* transposed K operand */
            acc += (double)q_row[c] * (double)k_head[c * N + j];
#else
            acc += (double)q_row[c] * (double)k_head[j * d + c];
#endif
        }
#if ORACLE_MUTANT == 1 /* dropped scale */
        s[j] = acc;
#else
        s[j] = scale * acc;
#endif
    }

    /* pass 1: row maximum */
    double m = -INFINITY;
    for (j = 0; j < N; ++j)
        if (s[j] > m)
            m = s[j];
    if (m == -INFINITY)
        m = 0.0; /* every score -inf: shift by 0, not (-inf) - (-inf) */

    /* pass 2: sum of shifted exponentials */
    double l = 0.0;
#if ORACLE_MUTANT == 5 /* off by one: last key dropped */
    for (j = 0; j + 1 < N; ++j)
#else
    for (j = 0; j < N; ++j)
#endif
    {
#if ORACLE_MUTANT == 3 /* wrong sign in the exponent */
        l += exp(m - s[j]);
#else
        l += exp(s[j] - m);
#endif
    }

    /* pass 3: normalised weights times V rows */
    for (c = 0; c < d; ++c)
        o_row[c] = 0.0;
    if (l == 0.0) { /* no key carries weight: O = 0, lse = -inf */
        *lse = -INFINITY;
        return;
    }
    for (j = 0; j < N; ++j) {
#if ORACLE_MUTANT == 3
        double w = exp(m - s[j]) / l;
#else
        double w = exp(s[j] - m) / l;
#endif
        for (c = 0; c < d; ++c) {
#if ORACLE_MUTANT == 6 /* transposed V operand */
            o_row[c] += w * (double)v_head[c * N + j];
#else
            o_row[c] += w * (double)v_head[j * d + c];
#endif
        }
    }

#if ORACLE_MUTANT == 4 /* log base 2 instead of natural log */
    *lse = m + log2(l);
#else
    *lse = m + log(l);
#endif
}

typedef struct {
    const float *q, *k, *v;
    int64_t B, H, H_kv, Nq, N, d; /* N = key/value rows per head */
    int causal;
    double scale;
    const int64_t *rows; /* nrows * 3 entries (b, h, i), or NULL = all */
    int64_t nrows;
    double *o, *lse;
    int64_t first, last; /* half-open range of output rows for a worker */
    int status;
} job_t;

static void *worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    double *s = (double *)malloc((size_t)(jb->N > 0 ? jb->N : 1) * sizeof(double));
    if (!s) {
        jb->status = -2;
        return NULL;
    }
    for (int64_t r = jb->first; r < jb->last; ++r) {
        int64_t b, h, i;
        if (jb->rows) {
            b = jb->rows[3 * r + 0];
            h = jb->rows[3 * r + 1];
            i = jb->rows[3 * r + 2];
        } else {
            i = r % jb->Nq;
            h = (r / jb->Nq) % jb->H;
            b = r / (jb->Nq * jb->H);
        }
        /* query head h reads key/value head h / (H / H_kv) */
        const int64_t kvh = b * jb->H_kv + h / (jb->H / jb->H_kv);
        const float *q_row = jb->q + ((b * jb->H + h) * jb->Nq + i) * jb->d;
        const int64_t kv_head = kvh * jb->N * jb->d;
        /* causal: query i sees the keys j <= i + (Nkv - Nq), a prefix of the
           key sequence; the other keys are excluded (weight 0) */
        int64_t visible = jb->N;
        if (jb->causal && i + (jb->N - jb->Nq) + 1 < visible)
            visible = i + (jb->N - jb->Nq) + 1;
        if (visible <= 0) { /* no visible key: O = 0, lse = -inf */
            for (int64_t c = 0; c < jb->d; ++c)
                jb->o[r * jb->d + c] = 0.0;
            jb->lse[r] = -INFINITY;
            continue;
        }
        attention_row(q_row, jb->k + kv_head, jb->v + kv_head,
                      visible, jb->d, jb->scale, s, jb->o + r * jb->d,
                      jb->lse + r);
    }
    free(s);
    return NULL;
}

/* Number of worker threads the oracle uses when asked for 0. */
int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Exact attention in fp64 for the selected rows, general shapes:
 *   q       : fp32 [B, H, Nq, d];   k, v : fp32 [B, H_kv, Nkv, d]
 *   query head h attends with key/value head h / (H / H_kv) (H_kv divides
 *   H; H_kv = H is plain multi-head attention).  Nq may differ from Nkv
 *   (Nq = 1: one decode step against Nkv cached keys, as in the FlashDecoding
 *   paragraph of "FlashAttention dissected", section "Interaction with the KV
 *   cache during inference").
 *   causal  : 0, or 1 for autoregressive attention: query i sees only keys
 *             j <= i + (Nkv - Nq) (the last query sees every key, as a decode
 *             step against a key cache does); a query with no visible key
 *             gets O = 0 and lse = -inf.  Not on the pages: the usual causal
 *             reading of the KV-cache paragraph of "FlashAttention dissected".
 *   rows    : NULL for every row (output order b, h, i), else nrows triples
 *             (b, h, i); out-of-range triples return -1.
 *   o       : fp64 [nrows, d];  lse : fp64 [nrows]
 *   threads : worker count, 0 = every online core.
 * Returns 0, or -1 on a bad argument, -2 when memory runs out.
 */
int oracle_attention_f64_ex(const float *q, const float *k, const float *v,
                            int64_t B, int64_t H, int64_t H_kv, int64_t Nq,
                            int64_t Nkv, int64_t d, double scale, int causal,
                            const int64_t *rows, int64_t nrows, double *o,
                            double *lse, int threads)
{
    if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 ||
        Nq < 1 || Nkv < 1 || d < 1)
        return -1;
    if (!rows)
        nrows = B * H * Nq;
    if (nrows < 0)
        return -1;
    if (rows) {
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t *t = rows + 3 * r;
            if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= H || t[2] < 0 || t[2] >= Nq)
                return -1;
        }
    }
    if (nrows == 0)
        return 0;
    if (threads <= 0)
        threads = oracle_default_threads();
    if ((int64_t)threads > nrows)
        threads = (int)nrows;

    job_t *jobs = (job_t *)calloc((size_t)threads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    for (int t = 0; t < threads; ++t) {
        job_t *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v;
        jb->B = B; jb->H = H; jb->H_kv = H_kv; jb->Nq = Nq; jb->N = Nkv; jb->d = d;
        jb->causal = causal;
        jb->scale = scale;
        jb->rows = rows;
        jb->nrows = nrows;
        jb->o = o; jb->lse = lse;
        jb->first = nrows * t / threads;
        jb->last = nrows * (t + 1) / threads;
        jb->status = 0;
    }
    int launched = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0)
            break;
        launched = t;
    }
    worker(&jobs[0]);
    /* rows of workers that could not be started run on this thread */
    for (int t = launched + 1; t < threads; ++t)
        worker(&jobs[t]);
    int status = jobs[0].status;
    for (int t = 1; t < threads; ++t) {
        if (t <= launched)
            pthread_join(tids[t], NULL);
        if (jobs[t].status != 0)
            status = jobs[t].status;
    }
    free(jobs);
    free(tids);
    return status;
}

/* Square self-attention form: q, k, v all [B, H, N, d]. */
int oracle_attention_f64(const float *q, const float *k, const float *v,
                         int64_t B, int64_t H, int64_t N, int64_t d,
                         double scale, const int64_t *rows, int64_t nrows,
                         double *o, double *lse, int threads)
{
    return oracle_attention_f64_ex(q, k, v, B, H, H, N, N, d, scale, 0, rows, nrows,
                                   o, lse, threads);
}

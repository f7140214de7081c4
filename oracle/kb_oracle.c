/*
 * kb_oracle.c -- fp64 CPU oracle for causal grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the GPU library is checked against.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (KernelBraid README, sections "Features" and
 * "Usage / Use a selected kernel"): BF16 causal attention over contiguous
 * [batch, heads, sequence, head_dim] tensors with 32 query heads sharing
 * 8 KV heads, head_dim 128.  For query row i of the block it is handed,
 * at absolute position p = start + i, the row attends to keys 0..p:
 *
 *     g      = h / (Hq / Hkv)                  (contiguous GQA groups)
 *     s_j    = (q[b,h,i,:] . k[b,g,j,:]) / sqrt(D),   j = 0..p
 *     o[b,h,i,:] = sum_j softmax(s)_j * v[b,g,j,:]
 *
 * Inputs are raw bf16 bit patterns; each is widened exactly to double.
 * Every product, sum, exp and the division are done in double, with the
 * row maximum subtracted before exp (this changes nothing mathematically).
 * Nothing here is blocked, fused or reordered: dot products and sums run
 * in ascending index order.
 *
 * Build: gcc -O2 -std=c11 -shared -fPIC -pthread kb_oracle.c -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact bf16 -> double: a bf16 value is the top 16 bits of an fp32. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int B, Hq, Hkv, Lq, D, start, cap;
    const int32_t *rows; /* n_rows triples (b, h, i) */
    int n_rows;
    double *out;         /* n_rows x D */
    int first, step;     /* this worker handles rows first, first+step, ... */
    int status;
} job_t;

/* One output row by the plain definition.  Returns 0 or a negative code. */
static int one_row(const job_t *J, int r, double *scores) {
    const int b = J->rows[3 * r + 0];
    const int h = J->rows[3 * r + 1];
    const int i = J->rows[3 * r + 2];
    if (b < 0 || b >= J->B || h < 0 || h >= J->Hq || i < 0 || i >= J->Lq) return -2;
    const int group = J->Hq / J->Hkv;
    const int g = h / group;
    const int p = J->start + i;      /* absolute position of this query row */
    const int ctx = p + 1;           /* keys 0..p are visible              */
    if (ctx > J->cap) return -3;
    const int D = J->D;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);

    const uint16_t *qrow = J->q + (((size_t)b * J->Hq + h) * J->Lq + i) * D;
    const uint16_t *kbase = J->k + ((size_t)b * J->Hkv + g) * (size_t)J->cap * D;
    const uint16_t *vbase = J->v + ((size_t)b * J->Hkv + g) * (size_t)J->cap * D;

    double qd[1024];
    for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(qrow[d]);

    double m = -INFINITY;
    for (int j = 0; j < ctx; ++j) {
        const uint16_t *krow = kbase + (size_t)j * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * bf16_to_double(krow[d]);
        scores[j] = dot * inv_sqrt_d;
        if (scores[j] > m) m = scores[j];
    }
    double denom = 0.0;
    for (int j = 0; j < ctx; ++j) {
        scores[j] = exp(scores[j] - m);
        denom += scores[j];
    }
    double *o = J->out + (size_t)r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int j = 0; j < ctx; ++j) {
        const uint16_t *vrow = vbase + (size_t)j * D;
        const double w = scores[j];
        for (int d = 0; d < D; ++d) o[d] += w * bf16_to_double(vrow[d]);
    }
    for (int d = 0; d < D; ++d) o[d] /= denom;
    return 0;
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(J->cap > 0 ? J->cap : 1));
    if (!scores) { J->status = -4; return NULL; }
    for (int r = J->first; r < J->n_rows; r += J->step) {
        int rc = one_row(J, r, scores);
        if (rc) { J->status = rc; break; }
    }
    free(scores);
    return NULL;
}

/*
 * kb_oracle_rows: attention for an explicit list of query rows.
 *
 *   q    bf16 bits [B][Hq][Lq][D]; row i sits at absolute position start+i
 *   k, v bf16 bits [B][Hkv][cap][D]; key rows 0..start+Lq-1 are read
 *   rows n_rows triples (b, h, i)
 *   out  double [n_rows][D]
 *
 * Returns 0, or -1 bad shape, -2 row index out of range, -3 context beyond
 * cap, -4 out of memory.
 */
int kb_oracle_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   int B, int Hq, int Hkv, int Lq, int D, int start, int cap,
                   const int32_t *rows, int n_rows, double *out, int n_threads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || D <= 0 || D > 1024 || start < 0 || cap <= 0)
        return -1;
    if (Hq % Hkv != 0) return -1;
    if (n_rows <= 0) return 0;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n_threads > n_rows) n_threads = n_rows;

    job_t jobs[256];
    pthread_t tids[256];
    for (int t = 0; t < n_threads; ++t) {
        job_t *J = &jobs[t];
        J->q = q; J->k = k; J->v = v;
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->Lq = Lq; J->D = D;
        J->start = start; J->cap = cap;
        J->rows = rows; J->n_rows = n_rows; J->out = out;
        J->first = t; J->step = n_threads; J->status = 0;
    }
    int created[256] = {0};
    for (int t = 1; t < n_threads; ++t)
        created[t] = (pthread_create(&tids[t], NULL, worker, &jobs[t]) == 0);
    worker(&jobs[0]);
    /* a worker that could not be started is run here instead */
    for (int t = 1; t < n_threads; ++t) {
        if (created[t]) pthread_join(tids[t], NULL);
        else worker(&jobs[t]);
    }
    for (int t = 0; t < n_threads; ++t)
        if (jobs[t].status) return jobs[t].status;
    return 0;
}

int kb_oracle_version(void) { return 1; }

/* ------------------------------------------------------------------------
 * Backward of the same attention (the gradient a training step needs).
 *
 * Causal prefill of a whole sequence (start = 0, every row 0..S-1).  With
 * P_i the softmax row above (keys 0..i), dO the gradient of the output and
 * 1/sqrt(D) the score scale:
 *
 *     dP_ij   = dO_i . v_j                        (j <= i)
 *     delta_i = sum_j P_ij dP_ij                  (the row's P . dP)
 *     dS_ij   = P_ij (dP_ij - delta_i)            (softmax Jacobian)
 *     dq_i    = sum_j dS_ij k_j / sqrt(D)
 *     dk_j    = sum over the group's query heads and rows i >= j of dS_ij q_i / sqrt(D)
 *     dv_j    = sum over the group's query heads and rows i >= j of P_ij dO_i
 *
 * All in double, loops in ascending index order.  Work is split by
 * (b, kv head), so the four query heads of a group add into dk, dv of that
 * unit alone and no two threads touch the same output.
 * ---------------------------------------------------------------------- */

typedef struct {
    const uint16_t *q, *k, *v, *dout;
    int B, Hq, Hkv, S, D;
    double *dq, *dk, *dv;   /* dq [B][Hq][S][D]; dk, dv [B][Hkv][S][D] */
    int first, step;        /* (b, g) units first, first+step, ... */
    int status;
} bwd_job_t;

/* Softmax row i of head h against keys 0..i: fills p[0..i] (normalised). */
static void softmax_row(const double *qd, const uint16_t *kbase, int i, int D, double inv_sqrt_d,
                        double *p) {
    double m = -INFINITY;
    for (int j = 0; j <= i; ++j) {
        const uint16_t *krow = kbase + (size_t)j * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * bf16_to_double(krow[d]);
        p[j] = dot * inv_sqrt_d;
        if (p[j] > m) m = p[j];
    }
    double denom = 0.0;
    for (int j = 0; j <= i; ++j) {
        p[j] = exp(p[j] - m);
        denom += p[j];
    }
    for (int j = 0; j <= i; ++j) p[j] /= denom;
}

static void *bwd_worker(void *arg) {
    bwd_job_t *J = (bwd_job_t *)arg;
    const int D = J->D, S = J->S, group = J->Hq / J->Hkv;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    double *p = (double *)malloc(sizeof(double) * (size_t)S);
    double *dp = (double *)malloc(sizeof(double) * (size_t)S);
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *dod = (double *)malloc(sizeof(double) * (size_t)D);
    if (!p || !dp || !qd || !dod) {
        J->status = -4;
        free(p); free(dp); free(qd); free(dod);
        return NULL;
    }
    for (int unit = J->first; unit < J->B * J->Hkv; unit += J->step) {
        const int b = unit / J->Hkv, g = unit % J->Hkv;
        const size_t kv_off = ((size_t)b * J->Hkv + g) * (size_t)S * D;
        const uint16_t *kbase = J->k + kv_off, *vbase = J->v + kv_off;
        double *dk = J->dk + kv_off, *dv = J->dv + kv_off;
        for (size_t e = 0; e < (size_t)S * D; ++e) { dk[e] = 0.0; dv[e] = 0.0; }
        for (int h = g * group; h < (g + 1) * group; ++h) {
            const size_t q_off = ((size_t)b * J->Hq + h) * (size_t)S * D;
            for (int i = 0; i < S; ++i) {
                const uint16_t *qrow = J->q + q_off + (size_t)i * D;
                const uint16_t *drow = J->dout + q_off + (size_t)i * D;
                for (int d = 0; d < D; ++d) { qd[d] = bf16_to_double(qrow[d]); dod[d] = bf16_to_double(drow[d]); }
                softmax_row(qd, kbase, i, D, inv_sqrt_d, p);
                double delta = 0.0;
                for (int j = 0; j <= i; ++j) {
                    const uint16_t *vrow = vbase + (size_t)j * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += dod[d] * bf16_to_double(vrow[d]);
                    dp[j] = dot;
                    delta += p[j] * dot;
                }
                double *dqrow = J->dq + q_off + (size_t)i * D;
                for (int d = 0; d < D; ++d) dqrow[d] = 0.0;
                for (int j = 0; j <= i; ++j) {
                    const double ds = p[j] * (dp[j] - delta);
                    const uint16_t *krow = kbase + (size_t)j * D;
                    double *dkrow = dk + (size_t)j * D, *dvrow = dv + (size_t)j * D;
                    for (int d = 0; d < D; ++d) {
                        dqrow[d] += ds * bf16_to_double(krow[d]) * inv_sqrt_d;
                        dkrow[d] += ds * qd[d] * inv_sqrt_d;
                        dvrow[d] += p[j] * dod[d];
                    }
                }
            }
        }
    }
    free(p); free(dp); free(qd); free(dod);
    return NULL;
}

static int run_threads(void *(*fn)(void *), void *jobs, size_t job_size, int n_threads) {
    pthread_t tids[256];
    int created[256] = {0};
    for (int t = 1; t < n_threads; ++t)
        created[t] = (pthread_create(&tids[t], NULL, fn, (char *)jobs + (size_t)t * job_size) == 0);
    fn(jobs);
    for (int t = 1; t < n_threads; ++t) {
        if (created[t]) pthread_join(tids[t], NULL);
        else fn((char *)jobs + (size_t)t * job_size);
    }
    return 0;
}

/*
 * kb_oracle_backward: dq, dk, dv of causal GQA attention over a whole
 * sequence (query row i at position i).
 *
 *   q, dout  bf16 bits [B][Hq][S][D];  k, v bf16 bits [B][Hkv][S][D]
 *   dq       double [B][Hq][S][D];     dk, dv double [B][Hkv][S][D]
 *
 * Returns 0, -1 bad shape, -4 out of memory.
 */
int kb_oracle_backward(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                       int B, int Hq, int Hkv, int S, int D, double *dq, double *dk, double *dv,
                       int n_threads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || D <= 0 || D > 1024 || Hq % Hkv != 0) return -1;
    const int units = B * Hkv;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n_threads > units) n_threads = units;
    bwd_job_t jobs[256];
    for (int t = 0; t < n_threads; ++t) {
        bwd_job_t *J = &jobs[t];
        J->q = q; J->k = k; J->v = v; J->dout = dout;
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->S = S; J->D = D;
        J->dq = dq; J->dk = dk; J->dv = dv;
        J->first = t; J->step = n_threads; J->status = 0;
    }
    run_threads(bwd_worker, jobs, sizeof(bwd_job_t), n_threads);
    for (int t = 0; t < n_threads; ++t)
        if (jobs[t].status) return jobs[t].status;
    return 0;
}

/* dq and the row statistics for listed rows (b, h, i) of a whole-sequence
 * prefill: dq_i as above, lse_i = log(sum_j exp(s_ij)) (natural log) and
 * delta_i = sum_j P_ij dP_ij.  Cost is one row's work per listed row. */
typedef struct {
    const uint16_t *q, *k, *v, *dout;
    int B, Hq, Hkv, S, D;
    const int32_t *rows;
    int n_rows;
    double *dq, *lse, *delta;  /* [n_rows][D], [n_rows], [n_rows] */
    int first, step;
    int status;
} dqrow_job_t;

static void *dqrow_worker(void *arg) {
    dqrow_job_t *J = (dqrow_job_t *)arg;
    const int D = J->D, S = J->S, group = J->Hq / J->Hkv;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)S);
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *dod = (double *)malloc(sizeof(double) * (size_t)D);
    if (!s || !qd || !dod) {
        J->status = -4;
        free(s); free(qd); free(dod);
        return NULL;
    }
    for (int r = J->first; r < J->n_rows; r += J->step) {
        const int b = J->rows[3 * r], h = J->rows[3 * r + 1], i = J->rows[3 * r + 2];
        if (b < 0 || b >= J->B || h < 0 || h >= J->Hq || i < 0 || i >= S) { J->status = -2; break; }
        const int g = h / group;
        const size_t q_off = (((size_t)b * J->Hq + h) * S + i) * D;
        const size_t kv_off = ((size_t)b * J->Hkv + g) * (size_t)S * D;
        for (int d = 0; d < D; ++d) { qd[d] = bf16_to_double(J->q[q_off + d]); dod[d] = bf16_to_double(J->dout[q_off + d]); }
        /* scores, max, normaliser */
        double m = -INFINITY;
        for (int j = 0; j <= i; ++j) {
            const uint16_t *krow = J->k + kv_off + (size_t)j * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qd[d] * bf16_to_double(krow[d]);
            s[j] = dot * inv_sqrt_d;
            if (s[j] > m) m = s[j];
        }
        double denom = 0.0;
        for (int j = 0; j <= i; ++j) denom += exp(s[j] - m);
        J->lse[r] = m + log(denom);
        /* P_ij = exp(s_ij - lse_i); delta, then dq */
        double delta = 0.0;
        for (int j = 0; j <= i; ++j) {
            const uint16_t *vrow = J->v + kv_off + (size_t)j * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += dod[d] * bf16_to_double(vrow[d]);
            const double p = exp(s[j] - m) / denom;
            s[j] = p;                      /* keep P_ij, and dP_ij below in place of the score */
            delta += p * dot;
        }
        J->delta[r] = delta;
        double *dqrow = J->dq + (size_t)r * D;
        for (int d = 0; d < D; ++d) dqrow[d] = 0.0;
        for (int j = 0; j <= i; ++j) {
            const uint16_t *vrow = J->v + kv_off + (size_t)j * D;
            const uint16_t *krow = J->k + kv_off + (size_t)j * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += dod[d] * bf16_to_double(vrow[d]);
            const double ds = s[j] * (dot - delta);
            for (int d = 0; d < D; ++d) dqrow[d] += ds * bf16_to_double(krow[d]) * inv_sqrt_d;
        }
    }
    free(s); free(qd); free(dod);
    return NULL;
}

int kb_oracle_dq_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                      int B, int Hq, int Hkv, int S, int D, const int32_t *rows, int n_rows,
                      double *dq, double *lse, double *delta, int n_threads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || D <= 0 || D > 1024 || Hq % Hkv != 0) return -1;
    if (n_rows <= 0) return 0;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n_threads > n_rows) n_threads = n_rows;
    dqrow_job_t jobs[256];
    for (int t = 0; t < n_threads; ++t) {
        dqrow_job_t *J = &jobs[t];
        J->q = q; J->k = k; J->v = v; J->dout = dout;
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->S = S; J->D = D;
        J->rows = rows; J->n_rows = n_rows; J->dq = dq; J->lse = lse; J->delta = delta;
        J->first = t; J->step = n_threads; J->status = 0;
    }
    run_threads(dqrow_worker, jobs, sizeof(dqrow_job_t), n_threads);
    for (int t = 0; t < n_threads; ++t)
        if (jobs[t].status) return jobs[t].status;
    return 0;
}

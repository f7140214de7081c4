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

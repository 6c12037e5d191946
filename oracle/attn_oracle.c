/*
 * FP64 CPU oracle for the dense, non-causal softmax attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it computes (the definition of standard attention: the dense BF16
 * attention that "Speed Up Image Generation with FLUX 3 Image Klein on NVIDIA
 * Blackwell GPUs", Key takeaways, second item, measures at about 60% of DiT
 * kernel time): for one query row i of head (b,h)
 *
 *     s_j = scale * sum_c q[i,c] * k[j,c]            j = 0 .. Lk-1
 *     m   = max_j s_j
 *     p_j = exp(s_j - m)
 *     l   = sum_j p_j
 *     o_c = (sum_j p_j * v[j,c]) / l
 *
 * Every step runs in double precision, in that order, with libm exp().
 * Inputs are either bfloat16 bit patterns (widened exactly to double) or
 * doubles.  Tensors are contiguous [B, H, L, d]; heads are addressed by the
 * flat index bh = b*H + h.  Build without -ffast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_BF16 = 0, ORACLE_F64 = 1 };

static double load_elem(const void *base, int kind, int64_t idx)
{
    if (kind == ORACLE_BF16) {
        uint32_t u = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return ((const double *)base)[idx];
}

typedef struct {
    const void *q, *k, *v;
    int kind;
    int64_t Lq, Lk, d;
    double scale;
    const int64_t *bh, *row;
    int64_t first, last;   /* rows [first, last) of the request */
    double *out;           /* [n_rows, d] */
    double *probs;         /* optional [n_rows, Lk]: p_j / l */
    int status;
} job_t;

static void *run_rows(void *arg)
{
    job_t *J = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)J->Lk);
    if (!s) { J->status = -1; return NULL; }
    for (int64_t r = J->first; r < J->last; ++r) {
        const int64_t bh = J->bh[r], i = J->row[r];
        const int64_t q0 = (bh * J->Lq + i) * J->d;
        const int64_t kv0 = bh * J->Lk * J->d;
        /* logits */
        for (int64_t j = 0; j < J->Lk; ++j) {
            double acc = 0.0;
            for (int64_t c = 0; c < J->d; ++c)
                acc += load_elem(J->q, J->kind, q0 + c) *
                       load_elem(J->k, J->kind, kv0 + j * J->d + c);
            s[j] = J->scale * acc;
        }
        /* max */
        double m = s[0];
        for (int64_t j = 1; j < J->Lk; ++j)
            if (s[j] > m) m = s[j];
        /* unnormalised probabilities and their sum */
        double l = 0.0;
        for (int64_t j = 0; j < J->Lk; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        /* weighted sum of values, divided by the sum */
        double *o = J->out + r * J->d;
        for (int64_t c = 0; c < J->d; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < J->Lk; ++j)
                acc += s[j] * load_elem(J->v, J->kind, kv0 + j * J->d + c);
            o[c] = acc / l;
        }
        if (J->probs) {
            double *p = J->probs + r * J->Lk;
            for (int64_t j = 0; j < J->Lk; ++j) p[j] = s[j] / l;
        }
    }
    free(s);
    return NULL;
}

/*
 * oracle_attention_rows: attention output for n_rows requested rows.
 *   q: [BH, Lq, d], k/v: [BH, Lk, d] (kind 0: uint16 bf16 bits, 1: double)
 *   bh[r], row[r]: flat head index and query row of request r
 *   out: [n_rows, d] doubles;  probs: NULL or [n_rows, Lk] (p_j / l)
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attention_rows(const void *q, const void *k, const void *v, int kind,
                          int64_t BH, int64_t Lq, int64_t Lk, int64_t d,
                          double scale, const int64_t *bh, const int64_t *row,
                          int64_t n_rows, double *out, double *probs, int n_threads)
{
    if (!q || !k || !v || !bh || !row || !out) return -1;
    if (BH < 1 || Lq < 1 || Lk < 1 || d < 1 || n_rows < 0) return -1;
    if (kind != ORACLE_BF16 && kind != ORACLE_F64) return -1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (bh[r] < 0 || bh[r] >= BH || row[r] < 0 || row[r] >= Lq) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_rows) n_threads = n_rows > 0 ? (int)n_rows : 1;

    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tid) { free(jobs); free(tid); return -1; }
    int status = 0;
    for (int t = 0; t < n_threads; ++t) {
        job_t *J = &jobs[t];
        J->q = q; J->k = k; J->v = v; J->kind = kind;
        J->Lq = Lq; J->Lk = Lk; J->d = d; J->scale = scale;
        J->bh = bh; J->row = row; J->out = out; J->probs = probs;
        J->first = n_rows * t / n_threads;
        J->last = n_rows * (t + 1) / n_threads;
    }
    int started = 0;
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tid[t], NULL, run_rows, &jobs[t]) != 0) { status = -1; break; }
        started = t;
    }
    run_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    if (status == 0 && started < n_threads - 1) status = -1;
    for (int t = 0; t < n_threads; ++t)
        if (jobs[t].status) status = -1;
    free(jobs);
    free(tid);
    return status;
}

/*
 * oracle_rmsnorm: y[r, c] = x[r, c] / sqrt(mean_c' x[r, c']^2 + eps) * w[c]
 * for every row r, in double precision (w = 1 when weight is NULL).
 *   x: [rows, d] (kind 0: uint16 bf16 bits, 1: double); weight: same kind or NULL
 *   y: [rows, d] doubles.  Returns 0, or -1 on bad arguments.
 * This is the per-token, per-head RMS normalisation of queries and keys that
 * the normalised workloads apply before attention.
 */
int oracle_rmsnorm(const void *x, const void *weight, int kind, int64_t rows, int64_t d,
                   double eps, double *y)
{
    if (!x || !y || rows < 1 || d < 1 || !(eps >= 0.0)) return -1;
    if (kind != ORACLE_BF16 && kind != ORACLE_F64) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            const double v = load_elem(x, kind, r * d + c);
            ss += v * v;
        }
        const double inv = 1.0 / sqrt(ss / (double)d + eps);
        for (int64_t c = 0; c < d; ++c) {
            const double w = weight ? load_elem(weight, kind, c) : 1.0;
            y[r * d + c] = load_elem(x, kind, r * d + c) * inv * w;
        }
    }
    return 0;
}

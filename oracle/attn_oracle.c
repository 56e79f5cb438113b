/*
 * attn_oracle.c -- plain fp64 CPU oracle for the attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes is the plain definition of the operation that the tiled
 * kernels replace ("OpenAI Triton: from introduction to model practice",
 * section 3, the PyTorch decoder layer: scores = Q K^T / sqrt(head_dim),
 * masked_fill of the causal mask, softmax over the key axis, then times V),
 * together with the per-row log-sum-exp that the FlashAttention rewrite in
 * section 5 of the same page stores next to O ("output + LSE", Figure 5 and
 * Source 2: lse = m_i + log(l_i), natural log, of the scaled scores).
 *
 * For every head (b, h) and query row i:
 *   J_i  = {0..N-1}, or {0..i} when causal            (masked keys excluded)
 *   s_j  = scale * sum_c q[i][c] * k[j][c]             for j in J_i
 *   m    = max_j s_j
 *   e_j  = exp(s_j - m),  l = sum_j e_j
 *   o[c] = sum_j e_j * v[j][c] / l
 *   lse  = m + ln(l)
 *
 * Two passes per row over a fully materialised score row; no tiling, no
 * online update.  Everything is double.  Inputs arrive as double arrays that
 * the caller upcast exactly from bf16.  Layout: contiguous [B][H][N][d], row
 * (b,h,i) starts at ((b*H + h)*N + i)*d.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEM 2

typedef struct {
    const double *q, *k, *v;
    double *o, *lse, *probs;
    int64_t H, N, d;
    double scale;
    int causal;
    const int64_t *rows; /* global row ids (b*H+h)*N+i, or NULL for all */
    int64_t row_begin, row_end;
    int status;
} oracle_job;

/* One query row, two passes over the materialised scores s[0..n_keys). */
static void one_row(const oracle_job *job, int64_t grow, int64_t out_idx, double *s)
{
    const int64_t N = job->N, d = job->d;
    const int64_t head = grow / N; /* b*H + h */
    const int64_t i = grow % N;
    const double *qi = job->q + grow * d;
    const double *kh = job->k + head * N * d;
    const double *vh = job->v + head * N * d;
    const int64_t n_keys = job->causal ? i + 1 : N; /* J_i = {0..n_keys-1} */

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) {
        const double *kj = kh + j * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += qi[c] * kj[c];
        s[j] = job->scale * dot;
        if (s[j] > m)
            m = s[j];
    }

    /* pass 2: exponentials, their sum, and the weighted sum of V rows */
    double *oi = job->o + out_idx * d;
    for (int64_t c = 0; c < d; ++c)
        oi[c] = 0.0;
    double l = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        const double e = exp(s[j] - m);
        s[j] = e;
        l += e;
        const double *vj = vh + j * d;
        for (int64_t c = 0; c < d; ++c)
            oi[c] += e * vj[c];
    }
    for (int64_t c = 0; c < d; ++c)
        oi[c] /= l;
    job->lse[out_idx] = m + log(l);

    if (job->probs) { /* full probability row, masked keys are exactly 0 */
        double *pi = job->probs + out_idx * N;
        for (int64_t j = 0; j < N; ++j)
            pi[j] = j < n_keys ? s[j] / l : 0.0;
    }
}

static void *run_job(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    double *s = (double *)malloc((size_t)(job->N > 0 ? job->N : 1) * sizeof(double));
    if (!s) {
        job->status = ORACLE_NO_MEM;
        return NULL;
    }
    for (int64_t r = job->row_begin; r < job->row_end; ++r) {
        const int64_t grow = job->rows ? job->rows[r] : r;
        one_row(job, grow, r, s);
    }
    free(s);
    job->status = ORACLE_OK;
    return NULL;
}

/*
 * oracle_attn_fwd: O and LSE for n_rows query rows.
 *   q,k,v   : double [B][H][N][d]
 *   rows    : n_rows global row ids in [0, B*H*N), or NULL meaning all rows
 *             in order (then n_rows must equal B*H*N)
 *   o       : double [n_rows][d]      (output)
 *   lse     : double [n_rows]         (output)
 *   probs   : double [n_rows][N] or NULL (output: the softmax row itself)
 *   threads : number of POSIX threads (>= 1)
 * Returns 0 on success.
 */
int oracle_attn_fwd(const double *q, const double *k, const double *v, double *o,
                    double *lse, double *probs, int64_t B, int64_t H, int64_t N,
                    int64_t d, double scale, int causal, const int64_t *rows,
                    int64_t n_rows, int threads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || n_rows < 0 || threads < 1)
        return ORACLE_BAD_ARG;
    if (n_rows == 0)
        return ORACLE_OK;
    if (!q || !k || !v || !o || !lse)
        return ORACLE_BAD_ARG;
    const int64_t total = B * H * N;
    if (!rows && n_rows != total)
        return ORACLE_BAD_ARG;
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total)
                return ORACLE_BAD_ARG;
    if (threads > n_rows)
        threads = (int)n_rows;

    oracle_job *jobs = (oracle_job *)calloc((size_t)threads, sizeof(oracle_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    char *running = (char *)calloc((size_t)threads, 1);
    if (!jobs || !tid || !running) {
        free(jobs);
        free(tid);
        free(running);
        return ORACLE_NO_MEM;
    }
    int status = ORACLE_OK;
    for (int t = 0; t < threads; ++t) {
        oracle_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->o = o; jb->lse = lse; jb->probs = probs;
        jb->H = H; jb->N = N; jb->d = d; jb->scale = scale; jb->causal = causal;
        jb->rows = rows;
        jb->row_begin = n_rows * t / threads;
        jb->row_end = n_rows * (t + 1) / threads;
        jb->status = ORACLE_BAD_ARG;
        if (threads > 1 && pthread_create(&tid[t], NULL, run_job, jb) == 0)
            running[t] = 1;
        else
            run_job(jb); /* one thread, or no thread could be started */
    }
    for (int t = 0; t < threads; ++t)
        if (running[t])
            pthread_join(tid[t], NULL);
    for (int t = 0; t < threads; ++t)
        if (jobs[t].status != ORACLE_OK)
            status = jobs[t].status;
    free(jobs);
    free(tid);
    free(running);
    return status;
}

/*
 * oracle_attn_fwd_kv: queries and keys of different lengths.
 *   q      : double [B][H][Nq][d]      k, v : double [B][H][Nk][d]
 *   o      : double [n_rows][d]        lse  : double [n_rows]
 *   rows   : global query rows (b*H + h)*Nq + i, or NULL for all B*H*Nq
 * The queries are the last Nq positions of the key sequence: under the
 * causal mask query i sees keys j <= i + (Nk - Nq) (requires Nq <= Nk);
 * without it, all Nk keys.  With Nq == Nk this is oracle_attn_fwd.
 * Same two-pass definition per row, in double.
 */
typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int64_t Nq, Nk, d;
    double scale;
    int causal;
    const int64_t *rows;
    int64_t row_begin, row_end;
    int status;
} oracle_kv_job;

static void *run_kv_job(void *arg)
{
    oracle_kv_job *jb = (oracle_kv_job *)arg;
    const int64_t Nq = jb->Nq, Nk = jb->Nk, d = jb->d;
    double *s = (double *)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    if (!s) {
        jb->status = ORACLE_NO_MEM;
        return NULL;
    }
    for (int64_t r = jb->row_begin; r < jb->row_end; ++r) {
        const int64_t grow = jb->rows ? jb->rows[r] : r;
        const int64_t head = grow / Nq, i = grow % Nq;
        const double *qi = jb->q + grow * d;
        const double *kh = jb->k + head * Nk * d;
        const double *vh = jb->v + head * Nk * d;
        const int64_t n_keys = jb->causal ? i + (Nk - Nq) + 1 : Nk;
        double m = -INFINITY;
        for (int64_t j = 0; j < n_keys; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += qi[c] * kh[j * d + c];
            s[j] = jb->scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        double *oi = jb->o + r * d;
        for (int64_t c = 0; c < d; ++c)
            oi[c] = 0.0;
        double l = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
            const double e = exp(s[j] - m);
            l += e;
            for (int64_t c = 0; c < d; ++c)
                oi[c] += e * vh[j * d + c];
        }
        for (int64_t c = 0; c < d; ++c)
            oi[c] /= l;
        jb->lse[r] = m + log(l);
    }
    free(s);
    jb->status = ORACLE_OK;
    return NULL;
}

int oracle_attn_fwd_kv(const double *q, const double *k, const double *v, double *o, double *lse,
                       int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, double scale,
                       int causal, const int64_t *rows, int64_t n_rows, int threads)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0 || n_rows < 0 || threads < 1)
        return ORACLE_BAD_ARG;
    if (causal && Nq > Nk)
        return ORACLE_BAD_ARG;
    if (n_rows == 0)
        return ORACLE_OK;
    if (!q || !k || !v || !o || !lse || Nk == 0)
        return ORACLE_BAD_ARG;
    const int64_t total = B * H * Nq;
    if (!rows && n_rows != total)
        return ORACLE_BAD_ARG;
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total)
                return ORACLE_BAD_ARG;
    if (threads > n_rows)
        threads = (int)n_rows;
    oracle_kv_job *jobs = (oracle_kv_job *)calloc((size_t)threads, sizeof(oracle_kv_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    char *running = (char *)calloc((size_t)threads, 1);
    if (!jobs || !tid || !running) {
        free(jobs);
        free(tid);
        free(running);
        return ORACLE_NO_MEM;
    }
    int status = ORACLE_OK;
    for (int t = 0; t < threads; ++t) {
        oracle_kv_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->o = o; jb->lse = lse;
        jb->Nq = Nq; jb->Nk = Nk; jb->d = d; jb->scale = scale; jb->causal = causal;
        jb->rows = rows;
        jb->row_begin = n_rows * t / threads;
        jb->row_end = n_rows * (t + 1) / threads;
        jb->status = ORACLE_BAD_ARG;
        if (threads > 1 && pthread_create(&tid[t], NULL, run_kv_job, jb) == 0)
            running[t] = 1;
        else
            run_kv_job(jb);
    }
    for (int t = 0; t < threads; ++t)
        if (running[t])
            pthread_join(tid[t], NULL);
    for (int t = 0; t < threads; ++t)
        if (jobs[t].status != ORACLE_OK)
            status = jobs[t].status;
    free(jobs);
    free(tid);
    free(running);
    return status;
}

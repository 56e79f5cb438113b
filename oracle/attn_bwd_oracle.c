/*
 * attn_bwd_oracle.c -- plain fp64 CPU oracle for the gradients of the
 * attention forward pass.  TEST INFRASTRUCTURE ONLY: nothing on the product
 * path calls, links or loads it, and it shares no code with the CUDA library.
 *
 * The forward pass is O = P V with P = softmax over visible keys of
 * S = scale * Q K^T ("OpenAI Triton: from introduction to model practice",
 * section 3).  Its gradients, given dO (the backward that section 6 of that
 * page wraps with the saved q, k, v, o, lse), are the chain rule written out:
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   D_i   = sum_j P_ij dP_ij            (= dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij K_j
 *   dK_j  = scale * sum_i dS_ij Q_i
 * with masked (causal) entries of P and dS equal to 0.  Everything is double,
 * in plain loops; P is recomputed from its definition (two passes per row).
 * Layout: contiguous [B][H][N][d] for q, k, v, dout and the outputs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *dout;
    double *dq, *dk, *dv;
    int64_t N, d;
    double scale;
    int causal;
    const int64_t *rows; /* dq-only mode: global row ids */
    int64_t begin, end;  /* heads (full mode) or row indices (dq-only mode) */
    int status;
} bwd_job;

/* P row i (visible keys) and dP row i; returns n_keys. */
static int64_t row_terms(const bwd_job *jb, const double *qh, const double *kh, const double *vh,
                         const double *doh, int64_t i, double *p, double *dp)
{
    const int64_t N = jb->N, d = jb->d;
    const int64_t n_keys = jb->causal ? i + 1 : N;
    const double *qi = qh + i * d, *doi = doh + i * d;
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += qi[c] * kh[j * d + c];
        p[j] = jb->scale * dot;
        if (p[j] > m)
            m = p[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int64_t j = 0; j < n_keys; ++j) {
        p[j] /= l;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += doi[c] * vh[j * d + c];
        dp[j] = dot;
    }
    return n_keys;
}

static void *run_full(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    const int64_t N = jb->N, d = jb->d;
    double *p = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *dp = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!p || !dp) {
        free(p);
        free(dp);
        jb->status = 2;
        return NULL;
    }
    for (int64_t h = jb->begin; h < jb->end; ++h) {
        const size_t off = (size_t)(h * N * d);
        const double *qh = jb->q + off, *kh = jb->k + off, *vh = jb->v + off, *doh = jb->dout + off;
        double *dqh = jb->dq + off, *dkh = jb->dk + off, *dvh = jb->dv + off;
        memset(dqh, 0, (size_t)(N * d) * sizeof(double));
        memset(dkh, 0, (size_t)(N * d) * sizeof(double));
        memset(dvh, 0, (size_t)(N * d) * sizeof(double));
        for (int64_t i = 0; i < N; ++i) {
            const int64_t n_keys = row_terms(jb, qh, kh, vh, doh, i, p, dp);
            double D = 0.0;
            for (int64_t j = 0; j < n_keys; ++j)
                D += p[j] * dp[j];
            for (int64_t j = 0; j < n_keys; ++j) {
                const double ds = p[j] * (dp[j] - D);
                for (int64_t c = 0; c < d; ++c) {
                    dvh[j * d + c] += p[j] * doh[i * d + c];
                    dqh[i * d + c] += jb->scale * ds * kh[j * d + c];
                    dkh[j * d + c] += jb->scale * ds * qh[i * d + c];
                }
            }
        }
    }
    free(p);
    free(dp);
    jb->status = 0;
    return NULL;
}

static void *run_dq_rows(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    const int64_t N = jb->N, d = jb->d;
    double *p = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *dp = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!p || !dp) {
        free(p);
        free(dp);
        jb->status = 2;
        return NULL;
    }
    for (int64_t r = jb->begin; r < jb->end; ++r) {
        const int64_t grow = jb->rows[r];
        const int64_t h = grow / N, i = grow % N;
        const size_t off = (size_t)(h * N * d);
        const double *qh = jb->q + off, *kh = jb->k + off, *vh = jb->v + off, *doh = jb->dout + off;
        const int64_t n_keys = row_terms(jb, qh, kh, vh, doh, i, p, dp);
        double D = 0.0;
        for (int64_t j = 0; j < n_keys; ++j)
            D += p[j] * dp[j];
        double *dqi = jb->dq + r * d;
        for (int64_t c = 0; c < d; ++c)
            dqi[c] = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
            const double ds = p[j] * (dp[j] - D);
            for (int64_t c = 0; c < d; ++c)
                dqi[c] += jb->scale * ds * kh[j * d + c];
        }
    }
    free(p);
    free(dp);
    jb->status = 0;
    return NULL;
}

/* dK and dV rows mode.  For one head at a time: first, for every query row
 * i of the head, the statistics of its softmax over the visible keys (max
 * m_i and sum l_i of exp(s_ij - m_i)) and D_i = sum_j P_ij dP_ij; then, for
 * each selected key j of that head, the sums over the query rows that see
 * it (i >= j under the causal mask):
 *   dV_j = sum_i P_ij dO_i,   dK_j = scale * sum_i P_ij (dP_ij - D_i) Q_i,
 * with P_ij = exp(s_ij - m_i) / l_i, s_ij = scale Q_i . K_j,
 * dP_ij = dO_i . V_j. */
typedef struct {
    const double *qh, *kh, *vh, *doh; /* the head's [N][d] blocks */
    double *m, *l, *D;                /* per query row of the head */
    double *dk, *dv;                  /* outputs [n_rows][d] */
    const int64_t *keys;              /* key index within the head, per output row */
    const int64_t *out_idx;           /* output row of each selected key */
    int64_t N, d;
    double scale;
    int causal;
    int64_t begin, end;
    int status;
} dkv_job;

static void *run_row_stats(void *arg)
{
    dkv_job *jb = (dkv_job *)arg;
    const int64_t N = jb->N, d = jb->d;
    double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!s) {
        jb->status = 2;
        return NULL;
    }
    for (int64_t i = jb->begin; i < jb->end; ++i) {
        const int64_t n_keys = jb->causal ? i + 1 : N;
        const double *qi = jb->qh + i * d, *doi = jb->doh + i * d;
        double m = -INFINITY;
        for (int64_t j = 0; j < n_keys; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += qi[c] * jb->kh[j * d + c];
            s[j] = jb->scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        double l = 0.0, acc = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
            const double e = exp(s[j] - m);
            double dp = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dp += doi[c] * jb->vh[j * d + c];
            l += e;
            acc += e * dp;
        }
        jb->m[i] = m;
        jb->l[i] = l;
        jb->D[i] = acc / l;
    }
    free(s);
    jb->status = 0;
    return NULL;
}

static void *run_key_rows(void *arg)
{
    dkv_job *jb = (dkv_job *)arg;
    const int64_t N = jb->N, d = jb->d;
    for (int64_t r = jb->begin; r < jb->end; ++r) {
        const int64_t j = jb->keys[r];
        double *dkj = jb->dk + jb->out_idx[r] * d, *dvj = jb->dv + jb->out_idx[r] * d;
        for (int64_t c = 0; c < d; ++c)
            dkj[c] = dvj[c] = 0.0;
        const double *kj = jb->kh + j * d, *vj = jb->vh + j * d;
        for (int64_t i = jb->causal ? j : 0; i < N; ++i) {
            const double *qi = jb->qh + i * d, *doi = jb->doh + i * d;
            double dot = 0.0, dp = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                dot += qi[c] * kj[c];
                dp += doi[c] * vj[c];
            }
            const double p = exp(jb->scale * dot - jb->m[i]) / jb->l[i];
            const double ds = p * (dp - jb->D[i]);
            for (int64_t c = 0; c < d; ++c) {
                dvj[c] += p * doi[c];
                dkj[c] += jb->scale * ds * qi[c];
            }
        }
    }
    jb->status = 0;
    return NULL;
}

static int run_dkv_jobs(dkv_job *proto, int64_t count, int threads, void *(*fn)(void *))
{
    if (count <= 0)
        return 0;
    if (threads > count)
        threads = (int)count;
    if (threads < 1)
        threads = 1;
    dkv_job *jobs = (dkv_job *)calloc((size_t)threads, sizeof(dkv_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    char *running = (char *)calloc((size_t)threads, 1);
    if (!jobs || !tid || !running) {
        free(jobs);
        free(tid);
        free(running);
        return 2;
    }
    for (int t = 0; t < threads; ++t) {
        jobs[t] = *proto;
        jobs[t].begin = count * t / threads;
        jobs[t].end = count * (t + 1) / threads;
        jobs[t].status = 1;
        if (threads > 1 && pthread_create(&tid[t], NULL, fn, &jobs[t]) == 0)
            running[t] = 1;
        else
            fn(&jobs[t]);
    }
    int status = 0;
    for (int t = 0; t < threads; ++t) {
        if (running[t])
            pthread_join(tid[t], NULL);
        if (jobs[t].status != 0)
            status = jobs[t].status;
    }
    free(jobs);
    free(tid);
    free(running);
    return status;
}

static int run_jobs(bwd_job *proto, int64_t count, int threads, void *(*fn)(void *))
{
    if (count <= 0)
        return 0;
    if (threads > count)
        threads = (int)count;
    if (threads < 1)
        threads = 1;
    bwd_job *jobs = (bwd_job *)calloc((size_t)threads, sizeof(bwd_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    char *running = (char *)calloc((size_t)threads, 1);
    if (!jobs || !tid || !running) {
        free(jobs);
        free(tid);
        free(running);
        return 2;
    }
    for (int t = 0; t < threads; ++t) {
        jobs[t] = *proto;
        jobs[t].begin = count * t / threads;
        jobs[t].end = count * (t + 1) / threads;
        jobs[t].status = 1;
        if (threads > 1 && pthread_create(&tid[t], NULL, fn, &jobs[t]) == 0)
            running[t] = 1;
        else
            fn(&jobs[t]);
    }
    int status = 0;
    for (int t = 0; t < threads; ++t) {
        if (running[t])
            pthread_join(tid[t], NULL);
        if (jobs[t].status != 0)
            status = jobs[t].status;
    }
    free(jobs);
    free(tid);
    free(running);
    return status;
}

/* Full gradients dq, dk, dv [B][H][N][d] of all heads. */
int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    double *dq, double *dk, double *dv, int64_t B, int64_t H, int64_t N, int64_t d,
                    double scale, int causal, int threads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0)
        return 1;
    if (B * H * N == 0)
        return 0;
    if (!q || !k || !v || !dout || !dq || !dk || !dv)
        return 1;
    bwd_job proto = {q, k, v, dout, dq, dk, dv, N, d, scale, causal, NULL, 0, 0, 0};
    return run_jobs(&proto, B * H, threads, run_full);
}

/* dq rows only, for the given global row ids (b*H + h)*N + i: dq_out [n_rows][d]. */
int oracle_attn_bwd_dq_rows(const double *q, const double *k, const double *v, const double *dout,
                            double *dq_out, int64_t B, int64_t H, int64_t N, int64_t d,
                            double scale, int causal, const int64_t *rows, int64_t n_rows,
                            int threads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || n_rows < 0)
        return 1;
    if (n_rows == 0)
        return 0;
    if (!q || !k || !v || !dout || !dq_out || !rows)
        return 1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N)
            return 1;
    bwd_job proto = {q, k, v, dout, dq_out, NULL, NULL, N, d, scale, causal, rows, 0, 0, 0};
    return run_jobs(&proto, n_rows, threads, run_dq_rows);
}

/* dk and dv rows only, for the given global KEY row ids (b*H + h)*N + j:
 * dk_out, dv_out [n_rows][d].  Each head that holds a selected key costs one
 * pass over all of its query rows (their softmax statistics and D_i). */
int oracle_attn_bwd_dkv_rows(const double *q, const double *k, const double *v,
                             const double *dout, double *dk_out, double *dv_out, int64_t B,
                             int64_t H, int64_t N, int64_t d, double scale, int causal,
                             const int64_t *rows, int64_t n_rows, int threads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || n_rows < 0)
        return 1;
    if (n_rows == 0)
        return 0;
    if (!q || !k || !v || !dout || !dk_out || !dv_out || !rows)
        return 1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N)
            return 1;
    double *stats = (double *)malloc((size_t)(3 * N) * sizeof(double));
    int64_t *keys = (int64_t *)malloc((size_t)n_rows * sizeof(int64_t));
    int64_t *out_idx = (int64_t *)malloc((size_t)n_rows * sizeof(int64_t));
    char *done = (char *)calloc((size_t)n_rows, 1);
    int status = (stats && keys && out_idx && done) ? 0 : 2;
    for (int64_t first = 0; status == 0 && first < n_rows; ++first) {
        if (done[first])
            continue;
        /* The selected keys of this head. */
        const int64_t h = rows[first] / N;
        int64_t count = 0;
        for (int64_t r = first; r < n_rows; ++r)
            if (!done[r] && rows[r] / N == h) {
                keys[count] = rows[r] % N;
                out_idx[count] = r;
                done[r] = 1;
                ++count;
            }
        const size_t off = (size_t)(h * N * d);
        dkv_job proto = {q + off, k + off, v + off, dout + off, stats, stats + N, stats + 2 * N,
                         dk_out, dv_out, keys, out_idx, N, d, scale, causal, 0, 0, 0};
        status = run_dkv_jobs(&proto, N, threads, run_row_stats);
        if (status == 0)
            status = run_dkv_jobs(&proto, count, threads, run_key_rows);
    }
    free(stats);
    free(keys);
    free(out_idx);
    free(done);
    return status;
}

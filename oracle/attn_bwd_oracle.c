/*
 * TEST INFRASTRUCTURE ONLY — the CPU oracle for the backward pass of exact attention.
 *
 * Only tests/ and bench.py's CPU-baseline leg load this library. The CUDA library never
 * links, includes or calls it, and it shares no code with the CUDA path.
 *
 * For one head the forward is o = softmax(q k^T / sqrt(d) + mask) v ("Flash attention in
 * PyTorch, then in Triton", "Attention's table of scores"). Given the gradient of the loss
 * with respect to the output, do, the page's section "Backwards, and training with it"
 * gives the gradients step by step, which this file follows in double precision with the
 * whole table of one head held in memory:
 *   1. S = q k^T * scale, masked entries excluded;  P = row softmax of S
 *   2. dV = P^T do
 *   3. dP = do v^T
 *   4. delta_i = sum_e do[i,e] * o[i,e]   (one number per row, formed once)
 *   5. dS = P * (dP - delta)  elementwise, per row (the softmax's backward)
 *   6. dQ = dS k * scale,  dK = dS^T q * scale (the scores carry the scale)
 * o in step 4 is this file's own forward (row softmax times v, in double), so nothing here
 * depends on a device result.
 *
 * Layout: q, k, v, do are float32 [B, H, N, d] holding the exact device values; dq, dk, dv
 * are double [B, H, N, d]. Heads run in parallel (pthreads); each head's arithmetic is
 * sequential, so the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    const float *q, *k, *v, *dout;
    int64_t N, d, BH;
    int causal;
    double *dq, *dk, *dv;
    int tid, nthreads, status;
} bwd_job;

static int head_backward(const float* q, const float* k, const float* v, const float* dout, int64_t N,
                         int64_t d, int causal, double* dq, double* dk, double* dv) {
    const double scale = 1.0 / sqrt((double)d);
    double* P = (double*)malloc(sizeof(double) * (size_t)(N * N));
    double* o = (double*)malloc(sizeof(double) * (size_t)d);
    double* dp = (double*)malloc(sizeof(double) * (size_t)N);
    if (!P || !o || !dp) {
        free(P);
        free(o);
        free(dp);
        return -2;
    }
    for (int64_t x = 0; x < N * d; ++x) dq[x] = dk[x] = dv[x] = 0.0;
    /* step 1: P, one row at a time (masked keys get weight 0) */
    for (int64_t i = 0; i < N; ++i) {
        const int64_t vis = causal ? i + 1 : N;
        double best = -HUGE_VAL;
        for (int64_t j = 0; j < N; ++j) {
            if (j >= vis) {
                P[i * N + j] = 0.0;
                continue;
            }
            double dot = 0.0;
            for (int64_t e = 0; e < d; ++e) dot += (double)q[i * d + e] * (double)k[j * d + e];
            P[i * N + j] = dot * scale;
            if (P[i * N + j] > best) best = P[i * N + j];
        }
        double total = 0.0;
        for (int64_t j = 0; j < vis; ++j) {
            P[i * N + j] = exp(P[i * N + j] - best);
            total += P[i * N + j];
        }
        for (int64_t j = 0; j < vis; ++j) P[i * N + j] /= total;
    }
    for (int64_t i = 0; i < N; ++i) {
        /* forward output of row i, then delta_i (step 4) */
        for (int64_t e = 0; e < d; ++e) o[e] = 0.0;
        for (int64_t j = 0; j < N; ++j)
            for (int64_t e = 0; e < d; ++e) o[e] += P[i * N + j] * (double)v[j * d + e];
        double delta = 0.0;
        for (int64_t e = 0; e < d; ++e) delta += (double)dout[i * d + e] * o[e];
        /* step 3: dP row i */
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t e = 0; e < d; ++e) acc += (double)dout[i * d + e] * (double)v[j * d + e];
            dp[j] = acc;
        }
        for (int64_t j = 0; j < N; ++j) {
            const double p = P[i * N + j];
            /* step 2: dV += P^T do */
            for (int64_t e = 0; e < d; ++e) dv[j * d + e] += p * (double)dout[i * d + e];
            /* step 5 */
            const double ds = p * (dp[j] - delta);
            /* step 6 */
            for (int64_t e = 0; e < d; ++e) {
                dq[i * d + e] += ds * (double)k[j * d + e] * scale;
                dk[j * d + e] += ds * (double)q[i * d + e] * scale;
            }
        }
    }
    free(P);
    free(o);
    free(dp);
    return 0;
}

static void* bwd_worker(void* arg) {
    bwd_job* job = (bwd_job*)arg;
    const int64_t head = job->N * job->d;
    job->status = 0;
    for (int64_t bh = job->tid; bh < job->BH; bh += job->nthreads) {
        const int st = head_backward(job->q + bh * head, job->k + bh * head, job->v + bh * head,
                                     job->dout + bh * head, job->N, job->d, job->causal, job->dq + bh * head,
                                     job->dk + bh * head, job->dv + bh * head);
        if (st != 0) {
            job->status = st;
            return NULL;
        }
    }
    return NULL;
}

/*
 * Gradients of exact attention with respect to q, k and v for the output gradient dout.
 *   q, k, v, dout : float32 [B, H, N, d]
 *   dq, dk, dv    : double [B, H, N, d]
 * Returns 0 on success, -1 on a bad argument, -2 when memory or threads run out.
 */
int oracle_attn_bwd(const float* q, const float* k, const float* v, const float* dout, int64_t B, int64_t H,
                    int64_t N, int64_t d, int causal, double* dq, double* dk, double* dv, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d <= 0 || (causal != 0 && causal != 1) || nthreads < 1) return -1;
    const int64_t BH = B * H;
    if (BH == 0 || N == 0) return 0;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
    if ((int64_t)nthreads > BH) nthreads = (int)BH;
    bwd_job* jobs = (bwd_job*)calloc((size_t)nthreads, sizeof(bwd_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    int started = 0, status = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (bwd_job){q, k, v, dout, N, d, BH, causal, dq, dk, dv, t, nthreads, -1};
        if (t == 0) continue;
        if (pthread_create(&th[t], NULL, bwd_worker, &jobs[t]) != 0) {
            status = -2;
            break;
        }
        started = t;
    }
    if (status == 0) bwd_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads && status == 0; ++t)
        if (jobs[t].status != 0) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

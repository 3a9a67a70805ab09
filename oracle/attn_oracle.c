/*
 * TEST INFRASTRUCTURE ONLY — the CPU oracle for exact attention forward.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference arm
 * load this library. The CUDA library never links, includes or calls it, and it shares
 * no code with the CUDA path.
 *
 * What it computes is the plain definition of scaled dot-product attention, as the
 * "Flash attention in PyTorch, then in Triton" page states it ("Attention's table of
 * scores", "Attention by hand"): for one head, scores are q_i . k_j / sqrt(d); under the
 * causal mask key j is visible to query i iff j <= i (the diagonal and the keys before
 * it); each row of visible scores goes through a softmax; the probabilities weigh the
 * value rows. The softmax is computed the way attention.cu's double-precision CPU
 * reference computes it ("CPU reference in double, one query row at a time, with the
 * maximum subtracted before any exp"): one row of scores is held, never the N x N matrix.
 *
 * Per query row i of head (b, h), in double:
 *   1. s_j = (sum_e q[i,e] * k[j,e]) * (1 / sqrt(d))   for every visible key j
 *   2. m   = max_j s_j
 *   3. w_j = exp(s_j - m),  L = sum_j w_j
 *   4. o[i,e] = (sum_j w_j * v[j,e]) / L
 *
 * The row's log-sum-exp, which the forward pass keeps for the backward pass, is the log of
 * the sum the softmax divides by. The page keeps it in base 2, as the running maximum plus
 * the base-2 log of the running total ("Backwards, and training with it"), i.e.
 * log2(sum_j exp(s_j)):
 *   5. lse2 = (m + log(L)) / ln(2)
 *
 * Inputs are float32 arrays that hold exactly the values the device reads (bf16/fp16
 * values widen to float32 exactly); every product and sum is in double. The only
 * parallelism is over independent rows (pthreads); each row's arithmetic is sequential
 * in key order, so the result does not depend on the thread count.
 *
 * Layout: q, k, v are [B, H, N, d] contiguous. Output rows are written in the order of
 * the requested row list, d doubles each.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const float* q;
    const float* k;
    const float* v;
    int64_t N, d, BH;
    int causal;
    const int64_t* rows; /* flat ids r = bh * N + i; NULL means all rows in order */
    int64_t nrows;
    double* o;
    double* lse; /* NULL, or one double per row */
    int tid, nthreads;
    int status;
} oracle_job;

/* One query row: fills o_row[0..d) and, if lse_row is not NULL, the row's base-2
 * log-sum-exp. s and acc are scratch of N and d doubles. */
static void oracle_row(const float* qh, const float* kh, const float* vh, int64_t N, int64_t d,
                       int causal, int64_t i, double* s, double* acc, double* o_row,
                       double* lse_row) {
    const double scale = 1.0 / sqrt((double)d);
    const int64_t visible = causal ? i + 1 : N;
    double best = -HUGE_VAL;
    for (int64_t j = 0; j < visible; ++j) {
        double dot = 0.0;
        for (int64_t e = 0; e < d; ++e) {
            dot += (double)qh[i * d + e] * (double)kh[j * d + e];
        }
        s[j] = dot * scale;
        if (s[j] > best) best = s[j];
    }
    double total = 0.0;
    for (int64_t j = 0; j < visible; ++j) {
        s[j] = exp(s[j] - best);
        total += s[j];
    }
    for (int64_t e = 0; e < d; ++e) acc[e] = 0.0;
    for (int64_t j = 0; j < visible; ++j) {
        const double w = s[j];
        for (int64_t e = 0; e < d; ++e) acc[e] += w * (double)vh[j * d + e];
    }
    for (int64_t e = 0; e < d; ++e) o_row[e] = acc[e] / total;
    if (lse_row) *lse_row = (best + log(total)) / log(2.0);
}

static void* oracle_worker(void* arg) {
    oracle_job* job = (oracle_job*)arg;
    double* s = (double*)malloc(sizeof(double) * (size_t)(job->N > 0 ? job->N : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)job->d);
    if (!s || !acc) {
        job->status = -2;
        free(s);
        free(acc);
        return NULL;
    }
    const int64_t head = job->N * job->d;
    /* Interleaved assignment balances the causal triangle across threads. */
    for (int64_t t = job->tid; t < job->nrows; t += job->nthreads) {
        const int64_t r = job->rows ? job->rows[t] : t;
        const int64_t bh = r / job->N;
        const int64_t i = r % job->N;
        oracle_row(job->q + bh * head, job->k + bh * head, job->v + bh * head, job->N, job->d,
                   job->causal, i, s, acc, job->o + t * job->d, job->lse ? job->lse + t : NULL);
    }
    free(s);
    free(acc);
    job->status = 0;
    return NULL;
}

/*
 * Exact attention forward for a list of query rows.
 *   q, k, v  : float32 [B, H, N, d] (host memory)
 *   rows     : flat row ids bh * N + i (0 <= bh < B*H, 0 <= i < N), or NULL for all rows
 *   nrows    : length of rows (ignored when rows is NULL: all B*H*N rows)
 *   o        : nrows x d doubles, row t holds the output of rows[t]
 *   lse      : NULL, or nrows doubles: lse[t] = log2 of the softmax denominator of rows[t]
 *   nthreads : worker threads (>= 1)
 * Returns 0 on success, -1 on a bad argument, -2 when memory or threads run out.
 */
int oracle_attn_fwd_lse(const float* q, const float* k, const float* v, int64_t B, int64_t H,
                        int64_t N, int64_t d, int causal, const int64_t* rows, int64_t nrows,
                        double* o, double* lse, int nthreads) {
    if (B < 0 || H < 0 || N < 0 || d <= 0 || (causal != 0 && causal != 1) || nthreads < 1)
        return -1;
    const int64_t BH = B * H;
    if (!rows) nrows = BH * N;
    if (nrows == 0) return 0;
    if (!q || !k || !v || !o) return -1;
    if (rows) {
        for (int64_t t = 0; t < nrows; ++t)
            if (rows[t] < 0 || rows[t] >= BH * N) return -1;
    }
    if ((int64_t)nthreads > nrows) nthreads = (int)nrows;
    oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    int started = 0, status = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (oracle_job){q, k, v, N, d, BH, causal, rows, nrows, o, lse, t, nthreads, -1};
        if (t == 0) continue; /* thread 0's share runs on the caller */
        if (pthread_create(&th[t], NULL, oracle_worker, &jobs[t]) != 0) {
            status = -2;
            break;
        }
        started = t;
    }
    if (status == 0) oracle_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads && status == 0; ++t)
        if (jobs[t].status != 0) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}

/* The same without log-sum-exps. */
int oracle_attn_fwd(const float* q, const float* k, const float* v, int64_t B, int64_t H,
                    int64_t N, int64_t d, int causal, const int64_t* rows, int64_t nrows,
                    double* o, int nthreads) {
    return oracle_attn_fwd_lse(q, k, v, B, H, N, d, causal, rows, nrows, o, NULL, nthreads);
}

/*
 * The normalised softmax weights of one query row of one head (steps 1-3 above, divided
 * by L): w[j] for j < N, zero for keys the causal mask hides. Used by tests to check that
 * each row of P sums to one and that masked keys get no weight.
 *   q, k : float32 [N, d] of one head;  w : N doubles.
 */
int oracle_attn_weights(const float* q, const float* k, int64_t N, int64_t d, int causal,
                        int64_t i, double* w) {
    if (!q || !k || !w || N <= 0 || d <= 0 || i < 0 || i >= N) return -1;
    const double scale = 1.0 / sqrt((double)d);
    const int64_t visible = causal ? i + 1 : N;
    double best = -HUGE_VAL;
    for (int64_t j = 0; j < N; ++j) w[j] = 0.0;
    for (int64_t j = 0; j < visible; ++j) {
        double dot = 0.0;
        for (int64_t e = 0; e < d; ++e) dot += (double)q[i * d + e] * (double)k[j * d + e];
        w[j] = dot * scale;
        if (w[j] > best) best = w[j];
    }
    double total = 0.0;
    for (int64_t j = 0; j < visible; ++j) {
        w[j] = exp(w[j] - best);
        total += w[j];
    }
    for (int64_t j = 0; j < visible; ++j) w[j] /= total;
    return 0;
}

/*
 * The key-value cache case: Nq new queries against Nk >= Nq keys, the queries being the last
 * Nq positions of the sequence. The "Flash attention in PyTorch, then in Triton" page names
 * this case (a handful of new tokens attending to every cached key, which its kernel leaves
 * out; section "Backwards, and training with it") without giving its mask; read plainly, query i sits at position Nk - Nq + i and, when causal, sees
 * the keys up to and including that position (all of the cache and the new tokens up to
 * itself). With Nq = Nk this is the ordinary causal mask. Per query row the arithmetic is
 * steps 1-5 above.
 *   q : float32 [B, H, Nq, d];  k, v : float32 [B, H, Nk, d]
 *   o : double [B, H, Nq, d];   lse : NULL or double [B, H, Nq] (base 2)
 */
int oracle_attn_fwd_kv(const float* q, const float* k, const float* v, int64_t B, int64_t H, int64_t Nq,
                       int64_t Nk, int64_t d, int causal, double* o, double* lse) {
    if (B < 0 || H < 0 || Nq < 0 || Nk < Nq || d <= 0 || (causal != 0 && causal != 1)) return -1;
    const int64_t BH = B * H;
    if (BH == 0 || Nq == 0) return 0;
    if (!q || !k || !v || !o) return -1;
    const double scale = 1.0 / sqrt((double)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !acc) {
        free(s);
        free(acc);
        return -2;
    }
    for (int64_t bh = 0; bh < BH; ++bh) {
        const float* qh = q + bh * Nq * d;
        const float* kh = k + bh * Nk * d;
        const float* vh = v + bh * Nk * d;
        for (int64_t i = 0; i < Nq; ++i) {
            const int64_t visible = causal ? (Nk - Nq + i + 1) : Nk;
            double best = -HUGE_VAL;
            for (int64_t j = 0; j < visible; ++j) {
                double dot = 0.0;
                for (int64_t e = 0; e < d; ++e) dot += (double)qh[i * d + e] * (double)kh[j * d + e];
                s[j] = dot * scale;
                if (s[j] > best) best = s[j];
            }
            double total = 0.0;
            for (int64_t j = 0; j < visible; ++j) {
                s[j] = exp(s[j] - best);
                total += s[j];
            }
            for (int64_t e = 0; e < d; ++e) acc[e] = 0.0;
            for (int64_t j = 0; j < visible; ++j)
                for (int64_t e = 0; e < d; ++e) acc[e] += s[j] * (double)vh[j * d + e];
            for (int64_t e = 0; e < d; ++e) o[(bh * Nq + i) * d + e] = acc[e] / total;
            if (lse) lse[bh * Nq + i] = (best + log(total)) / log(2.0);
        }
    }
    free(s);
    free(acc);
    return 0;
}

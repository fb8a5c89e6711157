/*
 * Exact attention forward -- plain, slow fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or constant
 * with the CUDA path.
 *
 * What it computes (the plain definition, written out):
 *   The pages describe the fused attention kernel as "scale, mask, softmax,
 *   weighted sum" done in one pass (zzycbzc.com/news/393333, section
 *   "算子融合的极致优化", item 2), and the standard implementation as the one
 *   that materialises the whole score matrix (same page, section
 *   "技术痛点").  Neither page writes the formula, so the oracle takes the
 *   plainest reading:
 *
 *     s_ij  = scale * sum_t q_it k_jt           for every allowed key j
 *     m_i   = max_j s_ij
 *     l_i   = sum_j exp(s_ij - m_i)
 *     O_i   = (sum_j exp(s_ij - m_i) v_j) / l_i
 *     LSE_i = m_i + ln(l_i)                      (natural log, scaled logits)
 *
 *   Allowed keys: all j when non-causal.  Causal ("causal": True, required
 *   for autoregressive models: 2kiu.com/news/1440730, section 3.2) allows
 *   key j for query i iff j <= i + (Nk - Nq); with Nq == Nk this is j <= i.
 *   A query row with no allowed key gets O = 0 and LSE = -inf.
 *
 *   This is the standard two-pass row algorithm (scores, then max and
 *   exponentials, then the weighted sum); it is deliberately NOT the online
 *   (running max / running sum) recurrence that the GPU path uses.
 *
 * Precision: inputs are given as fp64 (the caller upcasts the fp16/bf16
 * values exactly); every sum and exp/log is fp64.  Compiled with -O2 and
 * without fast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* Number of keys query row i may attend to. */
static long allowed_keys(long i, long Nq, long Nk, int causal)
{
    if (!causal) return Nk;
    long n = i + 1 + (Nk - Nq);
    if (n < 0) n = 0;
    if (n > Nk) n = Nk;
    return n;
}

/*
 * One query row.  q_row[d]; k_head, v_head: [Nk, d] row-major.
 * w: scratch of Nk doubles.  On return w[0..n) holds the unnormalised
 * weights exp(s_ij - m_i).  Returns n, the allowed-key count.
 */
static long attn_row(const double *q_row, const double *k_head,
                     const double *v_head, long i, long Nq, long Nk, long d,
                     int causal, double scale, double *o_row, double *lse,
                     double *w)
{
    long n = allowed_keys(i, Nq, Nk, causal);
    if (n == 0) {
        for (long t = 0; t < d; ++t) o_row[t] = 0.0;
        *lse = -INFINITY;
        return 0;
    }
    /* pass 1: scaled scores and their maximum */
    double m = -INFINITY;
    for (long j = 0; j < n; ++j) {
        const double *k_row = k_head + j * d;
        double dot = 0.0;
        for (long t = 0; t < d; ++t) dot += q_row[t] * k_row[t];
        double s = scale * dot;
        w[j] = s;
        if (s > m) m = s;
    }
    /* pass 2: exponentials relative to the maximum, and their sum */
    double l = 0.0;
    for (long j = 0; j < n; ++j) {
        double e = exp(w[j] - m);
        w[j] = e;
        l += e;
    }
    /* pass 3: weighted sum of values, normalised by the sum */
    for (long t = 0; t < d; ++t) {
        double acc = 0.0;
        for (long j = 0; j < n; ++j) acc += w[j] * v_head[j * d + t];
        o_row[t] = acc / l;
    }
    *lse = m + log(l);
    return n;
}

typedef struct {
    const double *q, *k, *v;
    long BH, Nq, Nk, d;
    int causal;
    double scale;
    const long *rows; /* NULL: every row */
    long nrows;
    double *o, *lse;
    long next;        /* next work item, shared */
    int running;      /* workers that got their scratch and take items */
    pthread_mutex_t lock;
} oracle_job;

static void *worker(void *arg)
{
    oracle_job *jb = (oracle_job *)arg;
    double *w = (double *)malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    if (!w) return NULL;   /* takes no items; another worker does them */
    pthread_mutex_lock(&jb->lock);
    jb->running += 1;
    pthread_mutex_unlock(&jb->lock);
    const long total = jb->BH * jb->nrows;
    const long chunk = 16;
    for (;;) {
        pthread_mutex_lock(&jb->lock);
        long begin = jb->next;
        jb->next += chunk;
        pthread_mutex_unlock(&jb->lock);
        if (begin >= total) break;
        long end = begin + chunk < total ? begin + chunk : total;
        for (long item = begin; item < end; ++item) {
            long bh = item / jb->nrows;
            long r = item % jb->nrows;
            long i = jb->rows ? jb->rows[r] : r;
            attn_row(jb->q + (bh * jb->Nq + i) * jb->d,
                     jb->k + bh * jb->Nk * jb->d,
                     jb->v + bh * jb->Nk * jb->d,
                     i, jb->Nq, jb->Nk, jb->d, jb->causal, jb->scale,
                     jb->o + item * jb->d, jb->lse + item, w);
        }
    }
    free(w);
    return NULL;
}

/*
 * Attention forward over BH independent (batch, head) problems.
 *   q: [BH, Nq, d]; k, v: [BH, Nk, d]; all row-major fp64.
 *   rows: NULL to compute every query row, else nrows query indices
 *         (the same subset for every head).
 *   o: [BH, nrows, d]; lse: [BH, nrows]   (nrows = Nq when rows is NULL)
 *   nthreads <= 0 uses one thread.
 * Returns 0 on success, -1 on bad arguments or when no worker could
 * allocate its scratch (then nothing was computed).
 */
int fa_oracle_fwd(const double *q, const double *k, const double *v,
                  long BH, long Nq, long Nk, long d, int causal, double scale,
                  const long *rows, long nrows, double *o, double *lse,
                  int nthreads)
{
    if (!q || !k || !v || !o || !lse) return -1;
    if (BH < 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    if (!rows) nrows = Nq;
    if (nrows < 0) return -1;
    if (rows)
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= Nq) return -1;
    if (BH == 0 || nrows == 0) return 0;
    if (nthreads < 1) nthreads = 1;

    oracle_job jb;
    jb.q = q; jb.k = k; jb.v = v;
    jb.BH = BH; jb.Nq = Nq; jb.Nk = Nk; jb.d = d;
    jb.causal = causal; jb.scale = scale;
    jb.rows = rows; jb.nrows = nrows;
    jb.o = o; jb.lse = lse;
    jb.next = 0;
    jb.running = 0;
    pthread_mutex_init(&jb.lock, NULL);

    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    if (tid)
        for (; started < nthreads; ++started)
            if (pthread_create(&tid[started], NULL, worker, &jb) != 0) break;
    if (started == 0) worker(&jb);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&jb.lock);
    /* any worker that started keeps taking items until none are left */
    return jb.running > 0 ? 0 : -1;
}

/*
 * Backward of the same attention, from the plain definition.  With
 * P = softmax(scale * Q K^T [mask]) and O = P V, for an upstream gradient
 * dO of O (the loss L = sum(O .* dO)):
 *   dV = P^T dO
 *   dP = dO V^T,   D_i = sum_t dO_it O_it
 *   dS = P .* (dP - D)          (the softmax Jacobian applied to dP)
 *   dQ = scale * dS K,   dK = scale * dS^T Q
 * computed row by row: each query row's P is built with the forward row
 * routine, dQ_i is finished at once, and dK, dV accumulate over the rows.
 * Rows are split into one chunk per thread, each with its own dK/dV partial
 * sums that are added at the end in chunk order (the result is the same for
 * a given thread count).
 */
typedef struct {
    const double *q, *k, *v, *dout;
    long Nq, Nk, d;
    int causal;
    double scale;
    long row0, row1;
    double *dq;               /* rows row0..row1 of dQ for this head */
    double *dk, *dv;          /* chunk-private [Nk, d] partial sums  */
    int failed;               /* set when the chunk could not run    */
} bwd_chunk;

static void *bwd_worker(void *arg)
{
    bwd_chunk *c = (bwd_chunk *)arg;
    const long d = c->d, Nk = c->Nk;
    double *w = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double *o_row = (double *)malloc(sizeof(double) * (size_t)d);
    if (!w || !o_row) { free(w); free(o_row); c->failed = 1; return NULL; }
    for (long i = c->row0; i < c->row1; ++i) {
        const double *qi = c->q + i * d, *gi = c->dout + i * d;
        double lse;
        long n = attn_row(qi, c->k, c->v, i, c->Nq, Nk, d, c->causal, c->scale,
                          o_row, &lse, w);
        double *dqi = c->dq + (i - c->row0) * d;
        for (long t = 0; t < d; ++t) dqi[t] = 0.0;
        if (n == 0) continue;
        double l = 0.0;
        for (long j = 0; j < n; ++j) l += w[j];
        double Di = 0.0;
        for (long t = 0; t < d; ++t) Di += gi[t] * o_row[t];
        for (long j = 0; j < n; ++j) {
            const double pj = w[j] / l;
            const double *vj = c->v + j * d, *kj = c->k + j * d;
            double dpj = 0.0;
            for (long t = 0; t < d; ++t) dpj += gi[t] * vj[t];
            const double dsj = pj * (dpj - Di);
            for (long t = 0; t < d; ++t) {
                c->dv[j * d + t] += pj * gi[t];
                c->dk[j * d + t] += c->scale * dsj * qi[t];
                dqi[t] += c->scale * dsj * kj[t];
            }
        }
    }
    free(w);
    free(o_row);
    return NULL;
}

/*
 * fa_oracle_bwd: gradients for BH independent problems.
 *   q, dout: [BH, Nq, d]; k, v: [BH, Nk, d]  ->  dq [BH, Nq, d],
 *   dk, dv [BH, Nk, d].  Returns 0, or -1 on bad arguments / no memory.
 */
int fa_oracle_bwd(const double *q, const double *k, const double *v,
                  const double *dout, long BH, long Nq, long Nk, long d,
                  int causal, double scale, double *dq, double *dk, double *dv,
                  int nthreads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
    if (BH < 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    if (nthreads < 1) nthreads = 1;
    const long nchunks = nthreads;
    bwd_chunk *ch = (bwd_chunk *)malloc(sizeof(bwd_chunk) * (size_t)nchunks);
    double *part = (double *)calloc((size_t)(2 * nchunks * (Nk > 0 ? Nk : 1) * d),
                                    sizeof(double));
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nchunks);
    if (!ch || !part || !tid) { free(ch); free(part); free(tid); return -1; }
    for (long h = 0; h < BH; ++h) {
        const long per = (Nq + nchunks - 1) / nchunks;
        for (long t = 0; t < nchunks; ++t) {
            bwd_chunk *c = &ch[t];
            c->q = q + h * Nq * d; c->dout = dout + h * Nq * d;
            c->k = k + h * Nk * d; c->v = v + h * Nk * d;
            c->Nq = Nq; c->Nk = Nk; c->d = d; c->causal = causal; c->scale = scale;
            c->row0 = t * per < Nq ? t * per : Nq;
            c->row1 = (t + 1) * per < Nq ? (t + 1) * per : Nq;
            c->dq = dq + (h * Nq + c->row0) * d;
            c->dk = part + (2 * t) * Nk * d;
            c->dv = part + (2 * t + 1) * Nk * d;
            c->failed = 0;
            memset(c->dk, 0, sizeof(double) * (size_t)(2 * Nk * d));
        }
        int started = 0;
        for (; started < nchunks; ++started)
            if (pthread_create(&tid[started], NULL, bwd_worker, &ch[started]) != 0) break;
        for (long t = started; t < nchunks; ++t) bwd_worker(&ch[t]);
        for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
        int failed = 0;
        for (long t = 0; t < nchunks; ++t) failed |= ch[t].failed;
        if (failed) { free(ch); free(part); free(tid); return -1; }
        double *dkh = dk + h * Nk * d, *dvh = dv + h * Nk * d;
        for (long e = 0; e < Nk * d; ++e) { dkh[e] = 0.0; dvh[e] = 0.0; }
        for (long t = 0; t < nchunks; ++t)
            for (long e = 0; e < Nk * d; ++e) {
                dkh[e] += ch[t].dk[e];
                dvh[e] += ch[t].dv[e];
            }
    }
    free(ch);
    free(part);
    free(tid);
    return 0;
}

/*
 * The normalised softmax weights p_ij = exp(s_ij - m_i) / l_i of one query
 * row i of one head, from the same row routine the forward uses.
 * p: Nk doubles; entries for masked keys are set to 0.
 * Returns the allowed-key count, or -1 on bad arguments.
 */
long fa_oracle_row_weights(const double *q_head, const double *k_head,
                           const double *v_head, long Nq, long Nk, long d,
                           int causal, double scale, long i, double *p)
{
    if (!q_head || !k_head || !v_head || !p || i < 0 || i >= Nq || d <= 0)
        return -1;
    double *o_row = (double *)malloc(sizeof(double) * (size_t)d);
    double *w = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    if (!o_row || !w) { free(o_row); free(w); return -1; }
    double lse;
    long n = attn_row(q_head + i * d, k_head, v_head, i, Nq, Nk, d, causal,
                      scale, o_row, &lse, w);
    double l = 0.0;
    for (long j = 0; j < n; ++j) l += w[j];
    for (long j = 0; j < Nk; ++j) p[j] = j < n ? w[j] / l : 0.0;
    free(o_row);
    free(w);
    return n;
}

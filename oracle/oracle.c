/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the attention forward and the
 * row-wise softmax / log-sum-exp.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through the seeded input generators.
 *
 * What it computes is the plain definition, not the online method:
 *
 *   softmax (three-pass "safe" form) -- "Softmax与Flash-Attention",
 *     section "safe-softmax 推导"; "什么是 online softmax and flash attention",
 *     section "Safe softmax", eq (2) and the three-pass listing after it;
 *     "从原始Softmax到在线Softmax", section "softmax形式推导":
 *         m = max_j x_j,   s = sum_j exp(x_j - m),   p_j = exp(x_j - m) / s.
 *
 *   log-sum-exp -- "从原始Softmax到在线Softmax", section "softmax形式推导"
 *     (the LSE(z) definition and log p_j = z_j - LSE(z)):
 *         LSE = m + log s        (natural logarithm).
 *
 *   attention -- "什么是 online softmax and flash attention", section
 *     "Attention的数学表达", eq (8)-(9) (Q[N,K], K[M,K], V[M,K], A[N,K]):
 *         x_j = scale * sum_k Q[i,k] K[j,k]     for every key j that is kept,
 *         O[i,:] = sum_j p_j V[j,:],            LSE[i] = m + log s.
 *     The causal mask keeps key j for query i iff j <= i (causal = 1, top-left
 *     aligned; the pages leave the mask's form open and this is the plainest
 *     reading) or iff j <= i + (M - N) (causal = 2, bottom-right aligned, the
 *     last query sees every key).  A query with no kept key has O = 0 and
 *     LSE = -inf (a convention: the definition is empty there).
 *
 * Every sum runs in index order in double precision; no blocking, fusion or
 * reordering.  Rows are independent, so they are spread over POSIX threads;
 * that changes which thread computes a row, never the arithmetic of a row.
 *
 * Layouts: X is [rows, cols] row-major.  Q is [B, H, N, d], K and V are
 * [B, H, M, d], all row-major, d fastest.  Attention outputs are produced for
 * a caller-chosen list of query rows given as flat indices (b*H + h)*N + i,
 * so that very large problems can be checked on a sample of rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Three-pass softmax of one row of n values; optional p and lse.     */
/* ------------------------------------------------------------------ */
static void softmax_three_pass(const double *x, long n, double *p, double *lse)
{
    /* pass 1: the maximum */
    double m = x[0];
    for (long j = 1; j < n; ++j)
        if (x[j] > m) m = x[j];
    /* pass 2: the sum of shifted exponentials */
    double s = 0.0;
    for (long j = 0; j < n; ++j)
        s += exp(x[j] - m);
    /* pass 3: the division */
    if (p)
        for (long j = 0; j < n; ++j)
            p[j] = exp(x[j] - m) / s;
    if (lse) *lse = m + log(s);
}

/* ------------------------------------------------------------------ */
/* Row-wise softmax / log-sum-exp                                     */
/* ------------------------------------------------------------------ */
typedef struct {
    const double *X;
    long rows, cols;
    double *P;     /* may be NULL */
    double *LSE;   /* may be NULL */
    long next;     /* shared work counter */
    pthread_mutex_t lock;
} rows_job;

static long take_row(long *next, pthread_mutex_t *lock, long limit)
{
    long r;
    pthread_mutex_lock(lock);
    r = *next;
    if (r < limit) *next = r + 1;
    pthread_mutex_unlock(lock);
    return r;
}

static void *rows_worker(void *arg)
{
    rows_job *job = (rows_job *)arg;
    for (;;) {
        long r = take_row(&job->next, &job->lock, job->rows);
        if (r >= job->rows) break;
        const double *x = job->X + r * job->cols;
        softmax_three_pass(x, job->cols,
                           job->P ? job->P + r * job->cols : NULL,
                           job->LSE ? job->LSE + r : NULL);
    }
    return NULL;
}

static int run_threads(void *(*fn)(void *), void *job, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tid) return -1;
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, fn, job) != 0) break;
        ++started;
    }
    fn(job);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    return 0;
}

/* Softmax probabilities (P, may be NULL) and natural-log LSE (may be NULL)
 * of each row of X[rows, cols].  Returns 0 on success, -1 on bad arguments. */
int oracle_softmax_rows(const double *X, long rows, long cols,
                        double *P, double *LSE, int nthreads)
{
    if (!X || rows < 0 || cols <= 0) return -1;
    rows_job job;
    job.X = X; job.rows = rows; job.cols = cols; job.P = P; job.LSE = LSE;
    job.next = 0;
    pthread_mutex_init(&job.lock, NULL);
    int rc = run_threads(rows_worker, &job, nthreads);
    pthread_mutex_destroy(&job.lock);
    return rc;
}

/* ------------------------------------------------------------------ */
/* Attention forward                                                  */
/* ------------------------------------------------------------------ */
typedef struct {
    const double *Q, *K, *V;
    long B, H, N, M, d;
    double scale;
    int causal;
    const long *sel;   /* selected flat query rows, or NULL for all */
    long nsel;
    double *O;         /* [nsel, d] */
    double *LSE;       /* [nsel], may be NULL */
    long next;
    pthread_mutex_t lock;
} attn_job;

static void *attn_worker(void *arg)
{
    attn_job *job = (attn_job *)arg;
    const long d = job->d, N = job->N, M = job->M;
    double *x = (double *)malloc(sizeof(double) * (size_t)M);
    double *p = (double *)malloc(sizeof(double) * (size_t)M);
    if (!x || !p) { free(x); free(p); return NULL; }
    for (;;) {
        long t = take_row(&job->next, &job->lock, job->nsel);
        if (t >= job->nsel) break;
        long flat = job->sel ? job->sel[t] : t;
        long bh = flat / N;             /* b*H + h */
        long i = flat % N;              /* query index within the head */
        const double *q = job->Q + flat * d;
        const double *Kh = job->K + bh * M * d;
        const double *Vh = job->V + bh * M * d;
        /* keys kept for this query: all M; 0..i under the top-left causal mask
         * (causal = 1); 0..i+(M-N) under the bottom-right one (causal = 2) */
        long kept = M;
        if (job->causal == 1 && i + 1 < M) kept = i + 1;
        if (job->causal == 2) {
            long last = i + (M - N);            /* last kept key */
            kept = last + 1 < M ? last + 1 : M;
            if (kept < 0) kept = 0;
        }
        double *o = job->O + t * d;
        if (kept == 0) {
            /* no key is kept: O = 0 and LSE = -inf by convention */
            for (long c = 0; c < d; ++c) o[c] = 0.0;
            if (job->LSE) job->LSE[t] = -INFINITY;
            continue;
        }
        /* materialise the score row x_j = scale * (q . k_j) */
        for (long j = 0; j < kept; ++j) {
            const double *k = Kh + j * d;
            double dot = 0.0;
            for (long c = 0; c < d; ++c) dot += q[c] * k[c];
            x[j] = job->scale * dot;
        }
        /* P = softmax(x) by the three passes, then O = P V */
        double lse;
        softmax_three_pass(x, kept, p, &lse);
        for (long c = 0; c < d; ++c) o[c] = 0.0;
        for (long j = 0; j < kept; ++j) {
            const double *v = Vh + j * d;
            for (long c = 0; c < d; ++c) o[c] += p[j] * v[c];
        }
        if (job->LSE) job->LSE[t] = lse;
    }
    free(x);
    free(p);
    return NULL;
}

/* Attention forward for a list of query rows.
 *   Q [B,H,N,d], K [B,H,M,d], V [B,H,M,d]  (fp64, row-major)
 *   sel: nsel flat query indices (b*H + h)*N + i, or NULL meaning all B*H*N
 *        rows in order (then nsel must equal B*H*N)
 *   O [nsel, d] out, LSE [nsel] out (may be NULL)
 * Returns 0 on success, -1 on bad arguments. */
int oracle_attn_rows(const double *Q, const double *K, const double *V,
                     long B, long H, long N, long M, long d,
                     double scale, int causal,
                     const long *sel, long nsel,
                     double *O, double *LSE, int nthreads)
{
    if (!Q || !K || !V || !O) return -1;
    if (B <= 0 || H <= 0 || N <= 0 || M <= 0 || d <= 0 || nsel < 0) return -1;
    if (causal < 0 || causal > 2) return -1;
    if (!sel && nsel != B * H * N) return -1;
    if (sel)
        for (long t = 0; t < nsel; ++t)
            if (sel[t] < 0 || sel[t] >= B * H * N) return -1;
    attn_job job;
    job.Q = Q; job.K = K; job.V = V;
    job.B = B; job.H = H; job.N = N; job.M = M; job.d = d;
    job.scale = scale; job.causal = causal;
    job.sel = sel; job.nsel = nsel; job.O = O; job.LSE = LSE;
    job.next = 0;
    pthread_mutex_init(&job.lock, NULL);
    int rc = run_threads(attn_worker, &job, nthreads);
    pthread_mutex_destroy(&job.lock);
    return rc;
}

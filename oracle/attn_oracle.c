/*
 * CPU fp64 oracle for exact scaled dot-product attention (test infrastructure).
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * may load this code. It shares nothing with the CUDA path: no headers, helpers,
 * constants or tables. It is plain and slow on purpose.
 *
 * What it computes, for one attention head, follows "Compilers and kernels"
 * (aaai.latere.ai/zh/infrastructure/compilers-kernels), section "FlashAttention
 * rewrites the algorithm around IO", first display and its symbol list:
 *
 *     S = Q K^T / sqrt(d) + C,   P_ij = exp(S_ij - m_i) / l_i,   O = P V,
 *     m_i = max_j S_ij,          l_i = sum_j exp(S_ij - m_i),
 *
 * with Q, K in R^{N x d}, V in R^{N x d_v}, C in (R u {-inf})^{N x N} additive
 * (-inf forbids a key) and at least one allowed key per row. The 1/sqrt(d) factor
 * is passed as `scale`; C is added after scaling and is not itself scaled.
 * LSE_i = m_i + ln l_i (natural log) is reported beside O.
 *
 * Readings where the pages are silent:
 *   - A row with no allowed key is excluded by the pages' assumption; the oracle
 *     defines O_i = 0 and LSE_i = -inf for it instead of dividing 0 by 0.
 *   - The additive C is the sum of the terms the mode bits select: CAUSAL gives
 *     -inf for key j > i + (Nk - Nq) and 0 otherwise (queries are the last Nq positions
 *     of the key sequence; for Nq = Nk this is j > i with shared indexing); DENSE reads
 *     C[bh][i][j]; KEY reads a per-key vector c[bh][j] (the same for every query row).
 *     No bit set means C = 0.
 *
 * The second, test-only path is the pages' blockwise online recurrence (same
 * section, the display for b_t, m_t, alpha_t, l_t, o_t and O_i = o_T / l_T) and
 * the three-quantity form of "AI Infra, ch. 5 Operators and runtime"
 * (pre.everytik.com/books/ai-infra/05), section 5.3 "FlashAttention", Example 5-6:
 * state (m, l, u), r = e^{m - m'}, l' = r l + p, u' = r u + p V, output u'/l'.
 *
 * All arithmetic is IEEE fp64 on the exact values of the bf16 / fp32 inputs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_NONE = 0, ORACLE_CAUSAL = 1, ORACLE_DENSE = 2, ORACLE_KEY = 4 };

/* Exact value of a bf16 bit pattern: the high half of an fp32. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *Q, *K, *V; /* bf16 bits, [BH][Nq][d], [BH][Nk][d], [BH][Nk][dv] */
    const float *C;            /* fp32 [BH][Nq][Nk] when the DENSE bit is set */
    const float *ckey;         /* fp32 [BH][Nk] when the KEY bit is set */
    int mode;                  /* bit set of CAUSAL, DENSE, KEY */
    int64_t BH, Nq, Nk, d, dv;
    double scale;
} problem_t;

/* C_ij of head bh: the sum of the terms the mode bits select. */
static double bias_value(const problem_t *p, int64_t bh, int64_t i, int64_t j)
{
    double c = 0.0;
    if ((p->mode & ORACLE_CAUSAL) && j > i + (p->Nk - p->Nq))
        return -INFINITY;
    if (p->mode & ORACLE_DENSE)
        c += (double)p->C[(bh * p->Nq + i) * p->Nk + j];
    if (p->mode & ORACLE_KEY)
        c += (double)p->ckey[bh * p->Nk + j];
    return c;
}

/*
 * One query row i of head bh, by the definition, with the whole row of S and P
 * materialised (S_row and P_row hold N doubles each):
 *   1. S_ij = scale * sum_k Q_ik K_jk + C_ij   for every key j
 *   2. m_i  = max_j S_ij
 *   3. l_i  = sum_j exp(S_ij - m_i)
 *   4. P_ij = exp(S_ij - m_i) / l_i
 *   5. O_i  = sum_j P_ij v_j
 *   6. LSE_i = m_i + ln l_i
 */
static void attention_row(const problem_t *p, int64_t bh, int64_t i, double *S_row,
                          double *P_row, double *O_row, double *lse)
{
    const int64_t N = p->Nk, d = p->d, dv = p->dv;
    const uint16_t *q = p->Q + (bh * p->Nq + i) * d;

    for (int64_t j = 0; j < N; j++) {
        const uint16_t *k = p->K + (bh * N + j) * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; c++)
            dot += bf16_value(q[c]) * bf16_value(k[c]);
        S_row[j] = p->scale * dot + bias_value(p, bh, i, j);
    }

    double m = -INFINITY;
    for (int64_t j = 0; j < N; j++)
        if (S_row[j] > m)
            m = S_row[j];

    if (m == -INFINITY) { /* no allowed key: outside the pages' assumption */
        for (int64_t j = 0; j < N; j++)
            P_row[j] = 0.0;
        for (int64_t c = 0; c < dv; c++)
            O_row[c] = 0.0;
        *lse = -INFINITY;
        return;
    }

    double l = 0.0;
    for (int64_t j = 0; j < N; j++)
        l += exp(S_row[j] - m);

    for (int64_t j = 0; j < N; j++)
        P_row[j] = exp(S_row[j] - m) / l;

    for (int64_t c = 0; c < dv; c++)
        O_row[c] = 0.0;
    for (int64_t j = 0; j < N; j++) {
        const uint16_t *v = p->V + (bh * N + j) * dv;
        for (int64_t c = 0; c < dv; c++)
            O_row[c] += P_row[j] * bf16_value(v[c]);
    }

    *lse = m + log(l);
}

typedef struct {
    const problem_t *p;
    const int64_t *rows; /* flat row ids bh * N + i; NULL means all rows */
    int64_t nrows;
    double *O;   /* [nrows][dv] */
    double *LSE; /* [nrows] */
    int64_t next;
    pthread_mutex_t lock;
} job_t;

static void *worker(void *arg)
{
    job_t *job = (job_t *)arg;
    const problem_t *p = job->p;
    double *S_row = (double *)malloc(sizeof(double) * (size_t)p->Nk);
    double *P_row = (double *)malloc(sizeof(double) * (size_t)p->Nk);
    if (!S_row || !P_row) {
        free(S_row);
        free(P_row);
        return (void *)1;
    }
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t r = job->next;
        job->next += 16;
        pthread_mutex_unlock(&job->lock);
        if (r >= job->nrows)
            break;
        int64_t end = r + 16 < job->nrows ? r + 16 : job->nrows;
        for (; r < end; r++) {
            int64_t flat = job->rows ? job->rows[r] : r;
            int64_t bh = flat / p->Nq, i = flat % p->Nq;
            attention_row(p, bh, i, S_row, P_row, job->O + r * p->dv, job->LSE + r);
        }
    }
    free(S_row);
    free(P_row);
    return NULL;
}

/*
 * Attention output rows by the definition, queries and keys of their own lengths.
 *   Q       : bf16 bit patterns, row-major [BH][Nq][d]
 *   K, V    : bf16 bit patterns, row-major [BH][Nk][d], [BH][Nk][dv]
 *   mode    : bit set: 1 CAUSAL (key j > i + Nk - Nq forbidden), 2 DENSE, 4 KEY
 *   C       : fp32 [BH][Nq][Nk] when DENSE is set (may hold -inf), else ignored
 *   ckey    : fp32 [BH][Nk] when KEY is set (may hold -inf), else ignored
 *   rows    : flat row ids (bh * Nq + i) to evaluate, or NULL for all BH * Nq rows
 *   O, LSE  : fp64 outputs, [nrows][dv] and [nrows], in the order of `rows`
 *   nthreads: worker threads; <= 0 means every online core
 * Returns the number of threads used, or -1 on bad arguments / allocation failure.
 */
int oracle_attention_ex(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int mode,
                        const float *C, const float *ckey, int64_t BH, int64_t Nq, int64_t Nk,
                        int64_t d, int64_t dv, double scale, const int64_t *rows, int64_t nrows,
                        double *O, double *LSE, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE || BH < 1 || Nq < 1 || Nk < 1 || d < 1 || dv < 1 ||
        nrows < 0)
        return -1;
    if (mode & ~(ORACLE_CAUSAL | ORACLE_DENSE | ORACLE_KEY))
        return -1;
    if (((mode & ORACLE_DENSE) && !C) || ((mode & ORACLE_KEY) && !ckey))
        return -1;
    if (!rows)
        nrows = BH * Nq;
    for (int64_t r = 0; rows && r < nrows; r++)
        if (rows[r] < 0 || rows[r] >= BH * Nq)
            return -1;

    problem_t p = {Q, K, V, C, ckey, mode, BH, Nq, Nk, d, dv, scale};
    job_t job;
    job.p = &p;
    job.rows = rows;
    job.nrows = nrows;
    job.O = O;
    job.LSE = LSE;
    job.next = 0;
    pthread_mutex_init(&job.lock, NULL);

    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    int64_t units = (nrows + 15) / 16;
    if (nthreads > units)
        nthreads = units > 0 ? (int)units : 1;

    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int failed = tid == NULL;
    int started = 0;
    for (int t = 0; !failed && t < nthreads; t++) {
        if (pthread_create(&tid[t], NULL, worker, &job) != 0)
            break;
        started++;
    }
    if (!failed && started == 0)
        failed = worker(&job) != NULL;
    for (int t = 0; t < started; t++) {
        void *ret = NULL;
        pthread_join(tid[t], &ret);
        failed |= ret != NULL;
    }
    free(tid);
    pthread_mutex_destroy(&job.lock);
    return failed ? -1 : (started > 0 ? started : 1);
}

/* The square problem (Nq = Nk = N) with mode NONE, CAUSAL or DENSE. */
int oracle_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int mode,
                     const float *C, int64_t BH, int64_t N, int64_t d, int64_t dv, double scale,
                     const int64_t *rows, int64_t nrows, double *O, double *LSE, int nthreads)
{
    if (mode != ORACLE_NONE && mode != ORACLE_CAUSAL && mode != ORACLE_DENSE)
        return -1;
    return oracle_attention_ex(Q, K, V, mode, C, NULL, BH, N, N, d, dv, scale, rows, nrows, O,
                               LSE, nthreads);
}

/*
 * The full score and probability matrices of one head (N x N each), with O and LSE,
 * by the same definition. For small N only: it materialises N^2 values twice.
 */
int oracle_attention_head(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int mode,
                          const float *C, int64_t N, int64_t d, int64_t dv, double scale,
                          double *S, double *P, double *O, double *LSE)
{
    if (!Q || !K || !V || !S || !P || !O || !LSE || N < 1 || d < 1 || dv < 1)
        return -1;
    if (mode == ORACLE_DENSE && !C)
        return -1;
    if (mode != ORACLE_NONE && mode != ORACLE_CAUSAL && mode != ORACLE_DENSE)
        return -1;
    problem_t p = {Q, K, V, C, NULL, mode, 1, N, N, d, dv, scale};
    for (int64_t i = 0; i < N; i++)
        attention_row(&p, 0, i, S + i * N, P + i * N, O + i * dv, LSE + i);
    return 0;
}

/*
 * The blockwise online recurrence for one query row (test-only second path).
 *   s      : scores S_ij of the row, n of them (forbidden keys may be -inf)
 *   v      : values, [n][dv]
 *   blk    : block index t in [0, T) of each key, or -1 for a key outside every block.
 *            The blocks B_1..B_T are meant to partition the allowed keys.
 *   order  : the order in which blocks are visited (a permutation of 0..T-1), or NULL
 * State: m_0 = -inf, l_0 = 0, o_0 = 0. For each block B_t in turn:
 *   b_t = max_{j in B_t} S_ij
 *   m_t = max(m_{t-1}, b_t)
 *   alpha_t = exp(m_{t-1} - m_t)
 *   l_t = alpha_t l_{t-1} + sum_{j in B_t} exp(S_ij - m_t)
 *   o_t = alpha_t o_{t-1} + sum_{j in B_t} exp(S_ij - m_t) v_j
 * Output: O_i = o_T / l_T, and the final m_T, l_T.
 * A block with no allowed key, visited before any allowed key, would give
 * exp(-inf - (-inf)); the pages' partition has no such block, and this function
 * returns -1 if it meets one.
 */
int oracle_online_blocks(const double *s, const double *v, int64_t n, int64_t dv,
                         const int *blk, int T, const int *order, double *O, double *m_out,
                         double *l_out)
{
    if (!s || !v || !blk || !O || n < 1 || dv < 1 || T < 1)
        return -1;
    double *o = (double *)calloc((size_t)dv, sizeof(double));
    if (!o)
        return -1;
    double m = -INFINITY, l = 0.0;
    for (int step = 0; step < T; step++) {
        int t = order ? order[step] : step;
        double b = -INFINITY;
        for (int64_t j = 0; j < n; j++)
            if (blk[j] == t && s[j] > b)
                b = s[j];
        double m_new = m > b ? m : b;
        if (m_new == -INFINITY) {
            free(o);
            return -1;
        }
        double alpha = exp(m - m_new);
        double block_sum = 0.0;
        for (int64_t c = 0; c < dv; c++)
            o[c] *= alpha;
        for (int64_t j = 0; j < n; j++) {
            if (blk[j] != t)
                continue;
            double e = exp(s[j] - m_new);
            block_sum += e;
            for (int64_t c = 0; c < dv; c++)
                o[c] += e * v[j * dv + c];
        }
        l = alpha * l + block_sum;
        m = m_new;
    }
    for (int64_t c = 0; c < dv; c++)
        O[c] = o[c] / l;
    free(o);
    if (m_out)
        *m_out = m;
    if (l_out)
        *l_out = l;
    return 0;
}

/*
 * One step of the three-quantity form: state (m, l, u) with u in R^{dv}, and one new
 * element with score s and value vector v (one element per block):
 *   m' = max(m, s),  r = e^{m - m'},  p = e^{s - m'},  l' = r l + p,  u' = r u + p v.
 * The caller reads the output as u' / l'. Updates the state in place.
 */
void oracle_online_step(double *m, double *l, double *u, int64_t dv, double s, const double *v)
{
    double m_new = *m > s ? *m : s;
    double r = exp(*m - m_new);
    double p = exp(s - m_new);
    *l = r * *l + p;
    for (int64_t c = 0; c < dv; c++)
        u[c] = r * u[c] + p * v[c];
    *m = m_new;
}

/*
 * Merge of two partial states (m1, l1, u1) and (m2, l2, u2) of disjoint key sets:
 * both are rescaled to the common maximum m = max(m1, m2) by the same alpha factor
 * the recurrence uses, then added. Both states must have seen at least one key.
 */
void oracle_online_merge(double m1, double l1, const double *u1, double m2, double l2,
                         const double *u2, int64_t dv, double *m, double *l, double *u)
{
    double mm = m1 > m2 ? m1 : m2;
    double a1 = exp(m1 - mm), a2 = exp(m2 - mm);
    *l = a1 * l1 + a2 * l2;
    for (int64_t c = 0; c < dv; c++)
        u[c] = a1 * u1[c] + a2 * u2[c];
    *m = mm;
}

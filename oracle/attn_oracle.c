/*
 * CPU fp64 oracle for exact scaled dot-product attention (test infrastructure).
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * may load this code. It shares nothing with the CUDA path: no headers, helpers,
 * constants or tables. It is plain and slow on purpose.
 *
 * What it computes, for one attention head, follows "Compilers and kernels", section
 * "FlashAttention rewrites the algorithm around IO", first display and its symbol list:
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
 * the three-quantity form of "AI Infra, ch. 5 Operators and runtime", section 5.3
 * "FlashAttention", Example 5-6:
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

/* ------------------------------------------------------------------------------
 * Backward pass (test infrastructure, like everything above).
 *
 * The pages state that the backward pass of the tiled method recomputes the local
 * score and probability blocks from Q, K and the kept softmax statistics instead of
 * storing them ("Compilers and kernels", section "FlashAttention rewrites the
 * algorithm around IO", the paragraph after the recurrence). The gradients themselves
 * are those of the forward display; for a loss whose gradient with respect to O is dO,
 * the chain rule through O = P V, the row softmax P = softmax(S) and
 * S = scale Q K^T + C gives
 *
 *     dV   = P^T dO
 *     dP   = dO V^T
 *     D_i  = sum_j P_ij dP_ij
 *     dS_ij = P_ij (dP_ij - D_i)        (the softmax Jacobian, row by row)
 *     dQ   = scale dS K,    dK = scale dS^T Q.
 *
 * The oracle evaluates them in two passes per head. Pass 1, per query row i: the row
 * of S and P by the definition (attention_row), the row of dP, D_i, and dQ_i; it keeps
 * m_i, l_i and D_i. Pass 2, per key j: S_ij and P_ij = exp(S_ij - m_i) / l_i for every
 * query row i again, then dV_j and dK_j. A row with no allowed key has P = 0, so it
 * contributes nothing (its output is the constant 0).
 * ------------------------------------------------------------------------------ */

typedef struct {
    const problem_t *p;
    const uint16_t *dO; /* bf16 bits [BH][Nq][dv] */
    int64_t bh;
    const int64_t *qrows; /* rows of this head for dQ, or NULL for all */
    int64_t nq_sel;
    const int64_t *krows; /* keys of this head for dK, dV, or NULL for all */
    int64_t nk_sel;
    double *m, *l, *D; /* [Nq] each: row max, row sum, D_i */
    double *dQ;        /* [nq_sel][d] */
    double *dK, *dV;   /* [nk_sel][d], [nk_sel][dv] */
    int pass;
    int64_t next, total;
    int failed;
    pthread_mutex_t lock;
} bwd_job_t;

/* Pass 1 for query row i: m_i, l_i, D_i, and dQ_i when `dq` is not NULL. */
static int bwd_row(const bwd_job_t *job, int64_t i, double *S_row, double *P_row, double *O_row,
                   double *dP_row, double *dq)
{
    const problem_t *p = job->p;
    const int64_t bh = job->bh, Nk = p->Nk, d = p->d, dv = p->dv;
    double lse;
    attention_row(p, bh, i, S_row, P_row, O_row, &lse);
    double m = -INFINITY;
    for (int64_t j = 0; j < Nk; j++)
        if (S_row[j] > m)
            m = S_row[j];
    double l = 0.0; /* l_i = sum_j exp(S_ij - m_i), kept for pass 2 */
    for (int64_t j = 0; m != -INFINITY && j < Nk; j++) {
        const double e = exp(S_row[j] - m);
        l += e;
    }
    job->m[i] = m;
    job->l[i] = l;

    const uint16_t *go = job->dO + (bh * p->Nq + i) * dv;
    double D = 0.0;
    for (int64_t j = 0; j < Nk; j++) {
        const uint16_t *v = p->V + (bh * Nk + j) * dv;
        double acc = 0.0;
        for (int64_t c = 0; c < dv; c++)
            acc += bf16_value(go[c]) * bf16_value(v[c]);
        dP_row[j] = acc;
        D += P_row[j] * acc;
    }
    job->D[i] = D;
    if (dq) {
        for (int64_t c = 0; c < d; c++)
            dq[c] = 0.0;
        for (int64_t j = 0; j < Nk; j++) {
            const double ds = P_row[j] * (dP_row[j] - D);
            const uint16_t *k = p->K + (bh * Nk + j) * d;
            for (int64_t c = 0; c < d; c++)
                dq[c] += ds * bf16_value(k[c]);
        }
        for (int64_t c = 0; c < d; c++)
            dq[c] *= p->scale;
    }
    return 0;
}

/* Pass 2 for key j: dK_j and dV_j over every query row of the head. */
static void bwd_key(const bwd_job_t *job, int64_t j, double *dk, double *dv_out)
{
    const problem_t *p = job->p;
    const int64_t bh = job->bh, Nk = p->Nk, d = p->d, dv = p->dv;
    const uint16_t *k = p->K + (bh * Nk + j) * d;
    const uint16_t *v = p->V + (bh * Nk + j) * dv;
    for (int64_t c = 0; c < d; c++)
        dk[c] = 0.0;
    for (int64_t c = 0; c < dv; c++)
        dv_out[c] = 0.0;
    for (int64_t i = 0; i < p->Nq; i++) {
        if (job->m[i] == -INFINITY)
            continue; /* no allowed key in row i: P_i = 0 */
        const uint16_t *q = p->Q + (bh * p->Nq + i) * d;
        const uint16_t *go = job->dO + (bh * p->Nq + i) * dv;
        double dot = 0.0;
        for (int64_t c = 0; c < d; c++)
            dot += bf16_value(q[c]) * bf16_value(k[c]);
        const double s = p->scale * dot + bias_value(p, bh, i, j);
        const double P = exp(s - job->m[i]) / job->l[i];
        double dP = 0.0;
        for (int64_t c = 0; c < dv; c++)
            dP += bf16_value(go[c]) * bf16_value(v[c]);
        const double ds = P * (dP - job->D[i]);
        for (int64_t c = 0; c < d; c++)
            dk[c] += ds * bf16_value(q[c]);
        for (int64_t c = 0; c < dv; c++)
            dv_out[c] += P * bf16_value(go[c]);
    }
    for (int64_t c = 0; c < d; c++)
        dk[c] *= p->scale;
}

static void *bwd_worker(void *arg)
{
    bwd_job_t *job = (bwd_job_t *)arg;
    const problem_t *p = job->p;
    const size_t n = (size_t)(p->Nk > p->dv ? p->Nk : p->dv);
    double *buf = (double *)malloc(sizeof(double) * (3 * (size_t)p->Nk + n));
    if (!buf) {
        pthread_mutex_lock(&job->lock);
        job->failed = 1;
        pthread_mutex_unlock(&job->lock);
        return NULL;
    }
    double *S_row = buf, *P_row = buf + p->Nk, *dP_row = buf + 2 * p->Nk, *O_row = buf + 3 * p->Nk;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t r = job->next;
        job->next += 8;
        pthread_mutex_unlock(&job->lock);
        if (r >= job->total)
            break;
        int64_t end = r + 8 < job->total ? r + 8 : job->total;
        for (; r < end; r++) {
            if (job->pass == 1) {
                /* every row i for m, l, D; dQ for the selected ones (pass 1 runs rows
                   in order, the selection is matched below) */
                bwd_row(job, r, S_row, P_row, O_row, dP_row, NULL);
            } else if (job->pass == 2) {
                int64_t i = job->qrows ? job->qrows[r] : r;
                bwd_row(job, i, S_row, P_row, O_row, dP_row, job->dQ + r * p->d);
            } else {
                int64_t j = job->krows ? job->krows[r] : r;
                bwd_key(job, j, job->dK + r * p->d, job->dV + r * p->dv);
            }
        }
    }
    free(buf);
    return NULL;
}

static int bwd_run(bwd_job_t *job, int pass, int64_t total, int nthreads)
{
    job->pass = pass;
    job->next = 0;
    job->total = total;
    int64_t units = (total + 7) / 8;
    if (nthreads > units)
        nthreads = units > 0 ? (int)units : 1;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; tid && t < nthreads; t++) {
        if (pthread_create(&tid[t], NULL, bwd_worker, job) != 0)
            break;
        started++;
    }
    if (started == 0)
        bwd_worker(job);
    for (int t = 0; t < started; t++)
        pthread_join(tid[t], NULL);
    free(tid);
    return started > 0 ? started : 1;
}

/*
 * Gradients dQ, dK, dV of the attention output for the loss gradient dO.
 *   Q, K, V, mode, C, ckey, BH, Nq, Nk, d, dv, scale: as oracle_attention_ex
 *   dO      : bf16 bit patterns, row-major [BH][Nq][dv]
 *   heads   : heads to evaluate (nheads of them), or NULL for all BH
 *   qrows   : query rows (within a head) whose dQ is wanted, or NULL for all Nq
 *   krows   : keys (within a head) whose dK and dV are wanted, or NULL for all Nk
 *   dQ      : fp64 [nheads][nq_sel][d];  dK: [nheads][nk_sel][d];  dV: [nheads][nk_sel][dv]
 *   nthreads: worker threads; <= 0 means every online core
 * Every head is evaluated on its own, rows and keys in a fixed order, so the result
 * does not depend on the thread count or on the selection.
 * Returns the number of threads used, or -1 on bad arguments / allocation failure.
 */
int oracle_attention_bwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                         const uint16_t *dO, int mode, const float *C, const float *ckey,
                         int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int64_t dv, double scale,
                         const int64_t *heads, int64_t nheads, const int64_t *qrows,
                         int64_t nq_sel, const int64_t *krows, int64_t nk_sel, double *dQ,
                         double *dK, double *dV, int nthreads)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV || BH < 1 || Nq < 1 || Nk < 1 || d < 1 ||
        dv < 1)
        return -1;
    if (mode & ~(ORACLE_CAUSAL | ORACLE_DENSE | ORACLE_KEY))
        return -1;
    if (((mode & ORACLE_DENSE) && !C) || ((mode & ORACLE_KEY) && !ckey))
        return -1;
    if (!heads)
        nheads = BH;
    if (!qrows)
        nq_sel = Nq;
    if (!krows)
        nk_sel = Nk;
    for (int64_t h = 0; heads && h < nheads; h++)
        if (heads[h] < 0 || heads[h] >= BH)
            return -1;
    for (int64_t r = 0; qrows && r < nq_sel; r++)
        if (qrows[r] < 0 || qrows[r] >= Nq)
            return -1;
    for (int64_t r = 0; krows && r < nk_sel; r++)
        if (krows[r] < 0 || krows[r] >= Nk)
            return -1;
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }

    problem_t p = {Q, K, V, C, ckey, mode, BH, Nq, Nk, d, dv, scale};
    double *stats = (double *)malloc(sizeof(double) * 3 * (size_t)Nq);
    if (!stats)
        return -1;
    bwd_job_t job;
    memset(&job, 0, sizeof job);
    job.p = &p;
    job.dO = dO;
    job.qrows = qrows;
    job.nq_sel = nq_sel;
    job.krows = krows;
    job.nk_sel = nk_sel;
    job.m = stats;
    job.l = stats + Nq;
    job.D = stats + 2 * Nq;
    pthread_mutex_init(&job.lock, NULL);
    int used = 1;
    for (int64_t h = 0; h < nheads; h++) {
        job.bh = heads ? heads[h] : h;
        job.dQ = dQ + h * nq_sel * d;
        job.dK = dK + h * nk_sel * d;
        job.dV = dV + h * nk_sel * dv;
        int u = bwd_run(&job, 1, Nq, nthreads); /* m, l, D of every row */
        used = u > used ? u : used;
        bwd_run(&job, 2, nq_sel, nthreads);     /* dQ of the selected rows */
        bwd_run(&job, 3, nk_sel, nthreads);     /* dK, dV of the selected keys */
    }
    pthread_mutex_destroy(&job.lock);
    free(stats);
    return job.failed ? -1 : used;
}

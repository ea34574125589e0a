/*
 * fp64 CPU oracle for exact scaled-dot-product attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is
 * compared against; it is not part of the product.  Only tests/,
 * __graft_entry__.smoke() and bench.py's CPU-baseline / reference leg may
 * load it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *   "FlashAttention: Part 2" (chizkidd.github.io), section 2.1 gives the
 *   function as softmax(Q K^T / sqrt(d)) V; section 6.2 ("FlashAttention
 *   Summary", "Ordinary attention" / "Naive execution") describes forming
 *   every score of a query row before the softmax; section 1.3 says one
 *   log-sum-exp value is kept per query row.  The scale is an argument
 *   (1/sqrt(d) in every workload here).
 *
 * For each requested row (b, hq, i):
 *   hkv      = hq / (Hq / Hkv)        -- contiguous GQA groups: the query
 *                                       heads hq = g*G .. g*G+G-1 share KV
 *                                       head g (pyshine.com flash-attention
 *                                       tour, "Why You Need This": K and V
 *                                       carry fewer heads, counts divide)
 *   L        = kv_len ? kv_len[b] : Nk
 *   visible(i, j) = (j < L) && (causal == 0 || j <= i + off)
 *            causal 1: aligned top-left, off = 0 (key j is seen by row i
 *                      iff j <= i);
 *            causal 2: aligned bottom-right, off = L - Nq (the last query
 *                      row sees every key; the pyshine.com flash-attention
 *                      tour, "Why You Need This", names this alignment)
 *            && (wl < 0 || j >= i + (L - Nq) - wl)
 *            && (wr < 0 || j <= i + (L - Nq) + wr)
 *                      local (sliding-window) attention, window (wl, wr):
 *                      row i sees keys no more than wl positions before it
 *                      and wr after it ("FlashAttention: Part 2", section
 *                      3.2: local attention keeps i -> j only for
 *                      |i - j| <= w; the pyshine.com tour, "From Install
 *                      to Causal Attention", passes the window as a
 *                      (left, right) pair next to causal).  Positions are
 *                      aligned bottom-right, as for causal 2; a negative
 *                      side is unbounded.
 *   s_j      = scale * sum_t q[i,t] * k[j,t]    (fp64; -inf if masked)
 *   m        = max_j s_j
 *   LSE      = m + ln(sum_j exp(s_j - m))       (natural log)
 *   P_j      = exp(s_j - LSE)
 *   O[t]     = sum_j P_j * v[j,t]
 * A row with no visible key returns O = 0 and LSE = -inf.
 *
 * Two passes over a fully materialised score row; no tiling, no online
 * recurrence, no blocking.  Inputs are bf16 bit patterns, widened exactly.
 * Layout is BSHD with d innermost:
 *   q[((b*Nq + i)*Hq + hq)*d + t]
 *   k[((b*Nk + j)*Hkv + hkv)*d + t]   (Nk = allocated key length)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int B, Hq, Hkv, Nq, Nk, d;
    const int32_t *kv_len;
    int causal;
    int wl, wr;
    double scale;
    const int32_t *rows; /* triples (b, hq, i) */
    int64_t n_rows;
    double *o;   /* n_rows * d */
    double *lse; /* n_rows */
    int n_threads;
    int thread_id;
    int status;
} oracle_job;

static void one_row(const oracle_job *J, int64_t r, double *s)
{
    const int b = J->rows[3 * r + 0];
    const int hq = J->rows[3 * r + 1];
    const int i = J->rows[3 * r + 2];
    const int d = J->d;
    const int group = J->Hq / J->Hkv;
    const int hkv = hq / group;
    const int L = J->kv_len ? J->kv_len[b] : J->Nk;
    const int off = (J->causal == 2) ? L - J->Nq : 0;
    const int64_t pos = (int64_t)i + L - J->Nq; /* row i's key position, bottom-right */
    const uint16_t *qrow = J->q + (((int64_t)b * J->Nq + i) * J->Hq + hq) * d;
    double *orow = J->o + r * d;

    /* pass 1: every score of the row, -inf where masked, and the row max */
    double m = -INFINITY;
    for (int j = 0; j < J->Nk; ++j) {
        int visible = (j < L) && (J->causal == 0 || j <= i + off) &&
                      (J->wl < 0 || j >= pos - J->wl) && (J->wr < 0 || j <= pos + J->wr);
        if (!visible) {
            s[j] = -INFINITY;
            continue;
        }
        const uint16_t *krow = J->k + (((int64_t)b * J->Nk + j) * J->Hkv + hkv) * d;
        double dot = 0.0;
        for (int t = 0; t < d; ++t)
            dot += bf16_value(qrow[t]) * bf16_value(krow[t]);
        s[j] = J->scale * dot;
        if (s[j] > m)
            m = s[j];
    }

    for (int t = 0; t < d; ++t)
        orow[t] = 0.0;
    if (m == -INFINITY) { /* no visible key */
        J->lse[r] = -INFINITY;
        return;
    }

    /* pass 2: denominator, then LSE */
    double sum = 0.0;
    for (int j = 0; j < J->Nk; ++j)
        if (s[j] != -INFINITY)
            sum += exp(s[j] - m);
    const double lse = m + log(sum);
    J->lse[r] = lse;

    /* pass 3: O = P V with P_j = exp(s_j - LSE) */
    for (int j = 0; j < J->Nk; ++j) {
        if (s[j] == -INFINITY)
            continue;
        const double p = exp(s[j] - lse);
        const uint16_t *vrow = J->v + (((int64_t)b * J->Nk + j) * J->Hkv + hkv) * d;
        for (int t = 0; t < d; ++t)
            orow[t] += p * bf16_value(vrow[t]);
    }
}

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->Nk > 0 ? J->Nk : 1));
    if (!s) {
        J->status = -2;
        return NULL;
    }
    for (int64_t r = J->thread_id; r < J->n_rows; r += J->n_threads)
        one_row(J, r, s);
    free(s);
    return NULL;
}

/*
 * Computes the rows listed in `rows` (n_rows triples b, hq, i).
 * window_left / window_right: the local window (negative: unbounded side).
 * Returns 0 on success, -1 on a bad argument, -2 on out-of-memory.
 */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d,
                     const int32_t *kv_len, int causal, int window_left, int window_right,
                     double scale,
                     const int32_t *rows, int64_t n_rows,
                     double *o, double *lse, int n_threads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0 || Hq % Hkv != 0)
        return -1;
    if (causal < 0 || causal > 2)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        const int32_t *t = rows + 3 * r;
        if (t[0] < 0 || t[0] >= B || t[1] < 0 || t[1] >= Hq || t[2] < 0 || t[2] >= Nq)
            return -1;
        if (kv_len && (kv_len[t[0]] < 0 || kv_len[t[0]] > Nk))
            return -1;
    }
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > 1024)
        n_threads = 1024;

    oracle_job *jobs = (oracle_job *)calloc((size_t)n_threads, sizeof(oracle_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return -2;
    }
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        oracle_job J = {q, k, v, B, Hq, Hkv, Nq, Nk, d, kv_len, causal, window_left, window_right, scale,
                        rows, n_rows, o, lse, n_threads, t, 0};
        jobs[t] = J;
    }
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tid[t], NULL, worker, &jobs[t]) != 0)
            break;
        started = t;
    }
    /* rows left to threads that failed to start are done here */
    if (started < n_threads - 1) {
        for (int t = started + 1; t < n_threads; ++t)
            worker(&jobs[t]);
    }
    worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tid[t], NULL);
    int status = 0;
    for (int t = 0; t < n_threads; ++t)
        if (jobs[t].status)
            status = jobs[t].status;
    free(jobs);
    free(tid);
    return status;
}

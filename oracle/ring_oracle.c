/*
 * ring_oracle.c -- plain, slow, fp64 CPU oracle for exact ring attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this library.  The product
 * path (the CUDA library under long_context_exact_ring_gb300/) never calls
 * it, and this file shares no code, header, table or constant with it.
 *
 * What it computes (all arithmetic in double precision, plain loops):
 *
 *   For one (batch b, head h) with Q, K, V in R^{S x d}, row-major, and the
 *   scaled score s_rc = scale * <q_r, k_c>:
 *     allowed set    A_r = { c : c <= r } when causal, else every c
 *     row maximum    M_r = max_{c in A_r} s_rc
 *     row LSE        LSE_r = M_r + ln sum_{c in A_r} exp(s_rc - M_r)
 *     output         O_r = sum_{c in A_r} exp(s_rc - LSE_r) v_c
 *
 *   That is the "exact" attention that Ring Attention reproduces
 *   ("Training Long-Context Models Without OOM: Ring Attention", section
 *   "Ring Attention Demystified": an exact mechanism that never forms the
 *   global s-by-s matrix).  The pages never print the softmax formula; the
 *   definition above is the textbook one.  Causal masking is not on the
 *   pages either; the reading taken is global-position masking c <= r.
 *
 * Two independent forward routines:
 *   oracle_naive_fwd   -- the definition over whole rows.
 *   oracle_ring_fwd    -- the ring schedule taken literally: the sequence is
 *                         split into P equal contiguous chunks (section
 *                         "Ring Attention Demystified", step 1; "Context
 *                         Parallelism" guide, section 2 "How It Works");
 *                         query chunk i visits KV chunk j = (i - t) mod P at
 *                         step t = 0..P-1 (step 0 local, later steps receive
 *                         from the left neighbour: steps 2-3 of the first
 *                         page, "Step 0 .. Step P-1" of the guide); each
 *                         visit yields a partial (O_ij, lse_ij) restricted
 *                         to chunk j, merged into a running pair with the
 *                         log-sum-exp merge ("running softmax normalization
 *                         statistics (the row maximum and running sum of
 *                         exponentials)", same section; "online softmax to
 *                         merge partial results", guide section 2).
 *
 * Backward (the pages only say activations are kept for the backward pass
 * and that recomputation trades compute for memory -- first page, sections
 * "Diagnosing the Sequence-Length OOM" and "Why the Parallelism You Already
 * Have Will Not Work"); the routine below is the plain derivative of the
 * definition for the loss L = sum(dO * O):
 *     P_rc = exp(s_rc - LSE_r) on A_r (0 elsewhere)
 *     dV = P^T dO,  dP = dO V^T,  D_r = sum_c P_rc dP_rc,
 *     dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_KIND_LOCAL 0 /* j == i: the query chunk's own KV chunk */
#define ORACLE_KIND_FULL 1  /* j != i and visited without a mask        */
#define ORACLE_KIND_SKIP 2  /* causal and j > i: contributes nothing    */

/* ------------------------------------------------------------------ */
/* Ring schedule                                                        */
/* ------------------------------------------------------------------ */

/* Visit list of query chunk i over the P ring steps t = 0..P-1.
 * out_j[t] = (i - t) mod P; out_kind[t] is LOCAL for t = 0, SKIP when
 * causal and j > i, FULL otherwise.  Returns P, or -1 on bad arguments. */
int oracle_ring_visits(int P, int causal, int i, int *out_j, int *out_kind)
{
    if (P < 1 || i < 0 || i >= P || !out_j || !out_kind)
        return -1;
    for (int t = 0; t < P; ++t) {
        int j = ((i - t) % P + P) % P;
        int kind;
        if (j == i)
            kind = ORACLE_KIND_LOCAL;
        else if (causal && j > i)
            kind = ORACLE_KIND_SKIP;
        else
            kind = ORACLE_KIND_FULL;
        out_j[t] = j;
        out_kind[t] = kind;
    }
    return P;
}

/* ------------------------------------------------------------------ */
/* Attention of one query row over a key range                          */
/* ------------------------------------------------------------------ */

static double dot(const double *a, const double *b, int d)
{
    double acc = 0.0;
    for (int x = 0; x < d; ++x)
        acc += a[x] * b[x];
    return acc;
}

/* Attention of query row q_r (global position r) over nk consecutive keys
 * Kb[0..nk), Vb[0..nk) whose global positions are c0, c0+1, ..., restricted
 * to positions <= r when causal.  Writes O (d values) and the natural-log
 * LSE.  An empty allowed set gives O = 0 and LSE = -inf (the identity of
 * the merge). */
static void attend_keys(const double *q_r, long r, const double *Kb,
                        const double *Vb, long c0, long nk, int d, int causal,
                        double scale, double *o_r, double *lse_r)
{
    long n = nk;
    if (causal && r - c0 + 1 < n)
        n = r - c0 + 1; /* keys at positions c0 .. r */
    for (int x = 0; x < d; ++x)
        o_r[x] = 0.0;
    if (n <= 0) {
        *lse_r = -INFINITY;
        return;
    }
    /* M_r */
    double m = -INFINITY;
    for (long c = 0; c < n; ++c) {
        double s = scale * dot(q_r, Kb + c * (long)d, d);
        if (s > m)
            m = s;
    }
    /* LSE_r = M_r + ln sum exp(s - M_r) */
    double sum = 0.0;
    for (long c = 0; c < n; ++c) {
        double s = scale * dot(q_r, Kb + c * (long)d, d);
        sum += exp(s - m);
    }
    double lse = m + log(sum);
    /* O_r = sum exp(s - LSE_r) v_c */
    for (long c = 0; c < n; ++c) {
        double s = scale * dot(q_r, Kb + c * (long)d, d);
        double p = exp(s - lse);
        const double *v_c = Vb + c * (long)d;
        for (int x = 0; x < d; ++x)
            o_r[x] += p * v_c[x];
    }
    *lse_r = lse;
}

/* Same, over the keys at positions [c_begin, c_end) of a whole head K, V. */
static void attend_row(const double *q_r, long r, const double *K,
                       const double *V, long c_begin, long c_end, int d,
                       int causal, double scale, double *o_r, double *lse_r)
{
    attend_keys(q_r, r, K + c_begin * (long)d, V + c_begin * (long)d, c_begin,
                c_end - c_begin, d, causal, scale, o_r, lse_r);
}

/* ------------------------------------------------------------------ */
/* Forward: the definition over whole rows                              */
/* ------------------------------------------------------------------ */

/* q, k, v: [B, H, S, d] row-major doubles.  o: [B, H, S, d]; lse: [B, H, S]. */
void oracle_naive_fwd(const double *q, const double *k, const double *v,
                      int B, int H, int S, int d, int causal, double scale,
                      double *o, double *lse)
{
    long total = (long)B * H * S;
#pragma omp parallel for schedule(dynamic, 16)
    for (long row = 0; row < total; ++row) {
        long bh = row / S;
        long r = row % S;
        const double *Kh = k + bh * (long)S * d;
        const double *Vh = v + bh * (long)S * d;
        attend_row(q + row * d, r, Kh, Vh, 0, S, d, causal, scale,
                   o + row * d, lse + row);
    }
}

/* Same definition, for an explicit list of rows: rows[n] is a flat row
 * index bh * S + r into the [B*H, S] grid.  o_rows: [nrows, d]. */
void oracle_naive_fwd_rows(const double *q, const double *k, const double *v,
                           int B, int H, int S, int d, int causal,
                           double scale, const int64_t *rows, long nrows,
                           double *o_rows, double *lse_rows)
{
    (void)B;
    (void)H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long n = 0; n < nrows; ++n) {
        long row = rows[n];
        long bh = row / S;
        long r = row % S;
        const double *Kh = k + bh * (long)S * d;
        const double *Vh = v + bh * (long)S * d;
        attend_row(q + row * d, r, Kh, Vh, 0, S, d, causal, scale,
                   o_rows + n * d, lse_rows + n);
    }
}

/* ------------------------------------------------------------------ */
/* The log-sum-exp merge of two partials                                */
/* ------------------------------------------------------------------ */

/* (O_a, lse_a) (+) (O_b, lse_b):
 *   m = max(lse_a, lse_b); w_a = exp(lse_a - m); w_b = exp(lse_b - m)
 *   O = (w_a O_a + w_b O_b) / (w_a + w_b);  lse = m + ln(w_a + w_b).
 * (0, -inf) is the identity; two -inf partials give (0, -inf). */
static void merge_pair(const double *o_a, double lse_a, const double *o_b,
                       double lse_b, int d, double *o_out, double *lse_out)
{
    double m = lse_a > lse_b ? lse_a : lse_b;
    if (m == -INFINITY) {
        for (int x = 0; x < d; ++x)
            o_out[x] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    double w_a = exp(lse_a - m);
    double w_b = exp(lse_b - m);
    double w = w_a + w_b;
    for (int x = 0; x < d; ++x)
        o_out[x] = (w_a * o_a[x] + w_b * o_b[x]) / w;
    *lse_out = m + log(w);
}

/* Row-wise merge over `rows` rows of width d.  The output may alias input
 * a: each element is read before it is written. */
void oracle_merge(const double *o_a, const double *lse_a, const double *o_b,
                  const double *lse_b, long rows, int d, double *o_out,
                  double *lse_out)
{
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r)
        merge_pair(o_a + r * d, lse_a[r], o_b + r * d, lse_b[r], d,
                   o_out + r * d, lse_out + r);
}

/* ------------------------------------------------------------------ */
/* Forward: the ring schedule, literally                                */
/* ------------------------------------------------------------------ */

/* S must be divisible by P.  visit_log (optional, P*P*3 ints) receives,
 * for query chunk i and step t, the triple (t, j, kind) at
 * visit_log[(i * P + t) * 3 + 0..2].  Returns 0, or -1 on bad arguments. */
int oracle_ring_fwd(const double *q, const double *k, const double *v,
                    int B, int H, int S, int d, int P, int causal,
                    double scale, double *o, double *lse, int *visit_log)
{
    if (P < 1 || S % P != 0 || d < 1 || d > 1024)
        return -1;
    long C = S / P;
    if (visit_log) {
        int js[4096], kinds[4096];
        if (P > 4096)
            return -1;
        for (int i = 0; i < P; ++i) {
            oracle_ring_visits(P, causal, i, js, kinds);
            for (int t = 0; t < P; ++t) {
                visit_log[(i * P + t) * 3 + 0] = t;
                visit_log[(i * P + t) * 3 + 1] = js[t];
                visit_log[(i * P + t) * 3 + 2] = kinds[t];
            }
        }
    }
    long total = (long)B * H * S;
#pragma omp parallel for schedule(dynamic, 16)
    for (long row = 0; row < total; ++row) {
        long bh = row / S;
        long r = row % S;
        int i = (int)(r / C);
        const double *Kh = k + bh * (long)S * d;
        const double *Vh = v + bh * (long)S * d;
        double o_run[1024], o_part[1024];
        double lse_run = -INFINITY; /* start from the identity (0, -inf) */
        for (int x = 0; x < d; ++x)
            o_run[x] = 0.0;
        for (int t = 0; t < P; ++t) {
            int j = ((i - t) % P + P) % P;
            if (causal && j > i)
                continue; /* the whole chunk lies above the diagonal */
            double lse_part;
            /* partial against chunk j; in chunk j == i the causal mask
             * c <= r applies inside attend_row, chunks j < i are full */
            attend_row(q + row * d, r, Kh, Vh, (long)j * C, (long)(j + 1) * C,
                       d, causal, scale, o_part, &lse_part);
            merge_pair(o_run, lse_run, o_part, lse_part, d, o_run, &lse_run);
        }
        memcpy(o + row * d, o_run, sizeof(double) * (size_t)d);
        lse[row] = lse_run;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Backward: the plain derivative of the definition                     */
/* ------------------------------------------------------------------ */

/* Full tensors.  Parallel over (b, h); within a head, plain loops over
 * query rows r and allowed keys c.  lse_out and d_out (optional, [B,H,S])
 * receive LSE_r and D_r. */
void oracle_bwd(const double *q, const double *k, const double *v,
                const double *dO, int B, int H, int S, int d, int causal,
                double scale, double *dq, double *dk, double *dv,
                double *lse_out, double *d_out)
{
    long BH = (long)B * H;
    memset(dq, 0, sizeof(double) * (size_t)(BH * S * d));
    memset(dk, 0, sizeof(double) * (size_t)(BH * S * d));
    memset(dv, 0, sizeof(double) * (size_t)(BH * S * d));
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh) {
        const double *Qh = q + bh * (long)S * d;
        const double *Kh = k + bh * (long)S * d;
        const double *Vh = v + bh * (long)S * d;
        const double *dOh = dO + bh * (long)S * d;
        double *dQh = dq + bh * (long)S * d;
        double *dKh = dk + bh * (long)S * d;
        double *dVh = dv + bh * (long)S * d;
        double *o_r = (double *)malloc(sizeof(double) * (size_t)d);
        double *Prow = (double *)malloc(sizeof(double) * (size_t)S);
        double *dProw = (double *)malloc(sizeof(double) * (size_t)S);
        for (long r = 0; r < S; ++r) {
            const double *q_r = Qh + r * d;
            const double *dO_r = dOh + r * d;
            double lse_r;
            attend_row(q_r, r, Kh, Vh, 0, S, d, causal, scale, o_r, &lse_r);
            long last = causal ? r + 1 : S;
            /* P_rc and dP_rc on the allowed set */
            for (long c = 0; c < last; ++c) {
                double s = scale * dot(q_r, Kh + c * (long)d, d);
                Prow[c] = exp(s - lse_r);
                dProw[c] = dot(dO_r, Vh + c * (long)d, d);
            }
            /* D_r = sum_c P_rc dP_rc */
            double D = 0.0;
            for (long c = 0; c < last; ++c)
                D += Prow[c] * dProw[c];
            for (long c = 0; c < last; ++c) {
                double dS = Prow[c] * (dProw[c] - D);
                const double *k_c = Kh + c * (long)d;
                double *dK_c = dKh + c * (long)d;
                double *dV_c = dVh + c * (long)d;
                for (int x = 0; x < d; ++x) {
                    dQh[r * d + x] += scale * dS * k_c[x];
                    dK_c[x] += scale * dS * q_r[x];
                    dV_c[x] += Prow[c] * dO_r[x];
                }
            }
            if (lse_out)
                lse_out[bh * S + r] = lse_r;
            if (d_out)
                d_out[bh * S + r] = D;
        }
        free(o_r);
        free(Prow);
        free(dProw);
    }
}

/* dQ for an explicit list of query rows (flat index bh * S + r).
 * Per row: LSE_r, P_rc, dP_rc, D_r, then dQ_r = scale sum_c dS_rc k_c.
 * Also returns D_r.  Cost O(S d) per row. */
void oracle_bwd_dq_rows(const double *q, const double *k, const double *v,
                        const double *dO, int B, int H, int S, int d,
                        int causal, double scale, const int64_t *rows,
                        long nrows, double *dq_rows, double *D_rows)
{
    (void)B;
    (void)H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long n = 0; n < nrows; ++n) {
        long row = rows[n];
        long bh = row / S;
        long r = row % S;
        const double *Kh = k + bh * (long)S * d;
        const double *Vh = v + bh * (long)S * d;
        const double *q_r = q + row * d;
        const double *dO_r = dO + row * d;
        double *out = dq_rows + n * d;
        double o_r[1024];
        double lse_r;
        attend_row(q_r, r, Kh, Vh, 0, S, d, causal, scale, o_r, &lse_r);
        long last = causal ? r + 1 : S;
        double D = 0.0;
        for (long c = 0; c < last; ++c) {
            double s = scale * dot(q_r, Kh + c * (long)d, d);
            D += exp(s - lse_r) * dot(dO_r, Vh + c * (long)d, d);
        }
        for (int x = 0; x < d; ++x)
            out[x] = 0.0;
        for (long c = 0; c < last; ++c) {
            double s = scale * dot(q_r, Kh + c * (long)d, d);
            double p = exp(s - lse_r);
            double dS = p * (dot(dO_r, Vh + c * (long)d, d) - D);
            const double *k_c = Kh + c * (long)d;
            for (int x = 0; x < d; ++x)
                out[x] += scale * dS * k_c[x];
        }
        D_rows[n] = D;
    }
}

/* ------------------------------------------------------------------ */
/* One ring step's partial, for rank-by-rank emulation                  */
/* ------------------------------------------------------------------ */

/* Partial attention of nq query rows (global positions r0 .. r0+nq-1)
 * against nk keys (global positions c0 .. c0+nk-1) of one head:
 * q_rows [nq, d], k_rows / v_rows [nk, d] -> o [nq, d], lse [nq].
 * Causal keeps c <= r.  A row with no allowed key gets (0, -inf). */
void oracle_partial(const double *q_rows, long r0, long nq,
                    const double *k_rows, const double *v_rows, long c0,
                    long nk, int d, int causal, double scale, double *o,
                    double *lse)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (long n = 0; n < nq; ++n)
        attend_keys(q_rows + n * d, r0 + n, k_rows, v_rows, c0, nk, d, causal,
                    scale, o + n * d, lse + n);
}

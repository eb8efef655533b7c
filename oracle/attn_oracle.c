/*
 * Exact-attention oracle: plain fp64 CPU implementation.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled and called by the tests, by
 * the package's smoke check and by the benchmark's CPU-baseline leg.  The GPU
 * product path never links or calls it, and it shares no code with the CUDA
 * sources.
 *
 * What it computes ("FlashAttention (HI)" page, section "Problems of standard
 * attention", formula Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V):
 *   for every query row (b, h, i) and every key j in the allowed set A(i)
 *     s_j   = scale * sum_t q[b,i,h,t] * k[b,j,h,t]
 *     O_i   = sum_j softmax(s)_j * v[b,j,h,:]
 *     lse_i = log sum_j exp(s_j)                    (natural log)
 *   A(i) = {0 .. N_k-1}; under the causal mask A(i) = {j <= i + N_k - N_q}
 *   (bottom-right alignment; equals j <= i when N_q == N_k).  A row with an
 *   empty A(i) gets O = 0 and lse = -inf.
 *
 * How ("FlashAttention (HI)" page, section "Online softmax computation"): one pass over the keys
 * that keeps a running maximum m, a running sum of exponentials l and a
 * running unnormalised output o, rescaling l and o whenever m grows:
 *   m' = max(m, s_j);  l = l e^{m-m'} + e^{s_j-m'};  o = o e^{m-m'} + e^{s_j-m'} v_j
 * then O = o / l and lse = m + log l.  No blocking, no reordering: keys are
 * visited in index order, and every quantity is a double.
 *
 * Layout: q, o are [B, N_q, H, d]; k, v are [B, N_k, H, d], row-major doubles.
 * lse is [B, H, N_q] for the full call and [n_rows] for the sampled call.
 *
 * ORACLE_MUTANT (compile-time, tests only) plants one known mistake so the
 * tests can show that the pins catch it; the normal build defines none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

static inline int64_t idx4(int64_t b, int64_t n, int64_t h, int64_t t,
                           int64_t N, int64_t H, int64_t d) {
    return ((b * N + n) * H + h) * d + t;
}

/* Last allowed key index for query row i (inclusive); -1 if none. */
static int64_t last_key(int64_t i, int64_t N_q, int64_t N_k, int causal) {
    if (!causal) return N_k - 1;
    int64_t lim = i + (N_k - N_q);
#if ORACLE_MUTANT == 4
    lim -= 1;                                   /* causal off-by-one */
#endif
    if (lim > N_k - 1) lim = N_k - 1;
    return lim < 0 ? -1 : lim;
}

/* One query row by the online recurrence.  acc is caller-provided, d doubles. */
static void one_row(const double* q, const double* k, const double* v,
                    int64_t b, int64_t h, int64_t i,
                    int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                    double scale, int causal, double* o_row, double* lse_out,
                    double* acc) {
    const double* qi = q + idx4(b, i, h, 0, N_q, H, d);
    int64_t jl = last_key(i, N_q, N_k, causal);
    double m = -INFINITY, l = 0.0;
    for (int64_t t = 0; t < d; ++t) acc[t] = 0.0;
    for (int64_t j = 0; j <= jl; ++j) {
#if ORACLE_MUTANT == 3
        const double* kj = k + idx4(b, j, (h + 1) % H, 0, N_k, H, d);  /* wrong head */
#else
        const double* kj = k + idx4(b, j, h, 0, N_k, H, d);
#endif
        const double* vj = v + idx4(b, j, h, 0, N_k, H, d);
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t) dot += qi[t] * kj[t];
#if ORACLE_MUTANT == 1
        double s = dot;                         /* scale dropped */
#else
        double s = scale * dot;
#endif
        double m_new = s > m ? s : m;
#if ORACLE_MUTANT == 2
        double alpha = exp(m_new - m);          /* wrong sign in the rescale */
#else
        double alpha = exp(m - m_new);          /* 0 when m = -inf */
#endif
        double p = exp(s - m_new);
#if ORACLE_MUTANT == 5
        l = l + p;                              /* sum not rescaled */
#else
        l = l * alpha + p;
#endif
        for (int64_t t = 0; t < d; ++t) acc[t] = acc[t] * alpha + p * vj[t];
        m = m_new;
    }
    if (jl < 0) {
        for (int64_t t = 0; t < d; ++t) o_row[t] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    for (int64_t t = 0; t < d; ++t) o_row[t] = acc[t] / l;
#if ORACLE_MUTANT == 6
    *lse_out = m + log(l) / scale;              /* lse in the wrong units */
#else
    *lse_out = m + log(l);
#endif
}

/* Sampled rows: rows is int64 [n_rows, 3] of (b, h, i); o is [n_rows, d]. */
int oracle_attn_rows(const double* q, const double* k, const double* v,
                     int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                     double scale, int causal,
                     const int64_t* rows, int64_t n_rows,
                     double* o, double* lse, int n_threads) {
    if (B <= 0 || H <= 0 || N_q < 0 || N_k < 0 || d <= 0) return 1;
    for (int64_t r = 0; r < n_rows; ++r) {
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 ||
            rows[3 * r + 1] >= H || rows[3 * r + 2] < 0 || rows[3 * r + 2] >= N_q)
            return 2;
    }
    int bad = 0;
#pragma omp parallel num_threads(n_threads > 0 ? n_threads : 1)
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!acc) {
#pragma omp atomic write
            bad = 3;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < n_rows; ++r)
                one_row(q, k, v, rows[3 * r], rows[3 * r + 1], rows[3 * r + 2],
                        H, N_q, N_k, d, scale, causal, o + r * d, lse + r, acc);
            free(acc);
        }
    }
    return bad;
}

/* Every row: o is [B, N_q, H, d], lse is [B, H, N_q]. */
int oracle_attn_full(const double* q, const double* k, const double* v,
                     int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                     double scale, int causal, double* o, double* lse, int n_threads) {
    if (B <= 0 || H <= 0 || N_q < 0 || N_k < 0 || d <= 0) return 1;
    int64_t total = B * H * N_q;
    int bad = 0;
#pragma omp parallel num_threads(n_threads > 0 ? n_threads : 1)
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!acc) {
#pragma omp atomic write
            bad = 3;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < total; ++r) {
                int64_t b = r / (H * N_q);
                int64_t h = (r / N_q) % H;
                int64_t i = r % N_q;
                one_row(q, k, v, b, h, i, H, N_q, N_k, d, scale, causal,
                        o + idx4(b, i, h, 0, N_q, H, d), lse + (b * H + h) * N_q + i, acc);
            }
            free(acc);
        }
    }
    return bad;
}

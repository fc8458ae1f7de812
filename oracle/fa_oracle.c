/*
 * Exact softmax attention, forward and backward, in double precision on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. This is the oracle that the CUDA path is checked
 * against. Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg load it; the library path never does, and the two share no code.
 *
 * What is computed, and where the definition comes from:
 *
 *  - Scores, softmax, output: "Why Flash Attention Is Fast: IO-Awareness
 *    Explained", section "Standard Attention's Real Bottleneck: HBM Access
 *    Count" (the three-step S = QK^T/sqrt(d), P = softmax(S), O = PV), and
 *    "FlashAttention Explained", section "A quick refresher on attention".
 *    The scale multiplies the raw dot products before the softmax, as in
 *    "FlashAttention" (deep dive), section "How it works" (S = Q K^T * scale).
 *  - Logsumexp per row, natural log, L = m + log l: "FlashAttention" (deep
 *    dive), section "How it works", and its Rust listing's comment that L is all
 *    the backward pass needs.  Here it is written out as L_i = M_i + ln Z_i with
 *    M_i the row maximum of the scaled scores and Z_i = sum_j exp(S_ij - M_i).
 *  - Causal masking: "tm_flash_attention_arch_2k", section "The architecture:
 *    every step explained" (upper-triangular positions have no effect).  Read as
 *    the square, top-left aligned mask: key j is visible to query i iff j <= i.
 *  - Backward: "FlashAttention" (deep dive), section "How it works":
 *    D = rowsum(dO o O), dS = P o (dP - D).  With S carrying the scale, the chain
 *    rule gives dV = P^T dO, dP = dO V^T, dQ = scale * dS K, dK = scale * dS^T Q.
 *    Masked entries have P = 0 and therefore dS = 0.
 *  - A row with no visible key ("FlashAttention" deep dive, section "Pitfalls":
 *    output 0) gets O = 0 and L = -inf.  With N >= 1 and the top-left causal mask
 *    every row sees key 0, so this case is unreachable through the public entry
 *    points; it is kept so that the definition is total.
 *
 * Everything is the plain definition: one query row at a time, its full row of
 * scores materialised, no tiling, no online rescaling.  Loops over (head, row)
 * run in parallel with OpenMP; each output element is written by one thread.
 *
 * Layout: every tensor is [B, H, N, d] contiguous (row stride d, head stride
 * N*d); L is [B, H, N].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Number of keys query row i may see. */
static long visible_keys(long i, long n, int causal) {
    return causal ? (i + 1 < n ? i + 1 : n) : n;
}

/*
 * One query row: scaled scores against the visible keys, then the softmax
 * probabilities p[0..nk) and the logsumexp.  Returns nk (0 means no key).
 */
static long softmax_row(const double *qi, const double *kh, long i, long n, long d,
                        double scale, int causal, double *p, double *lse_out) {
    long nk = visible_keys(i, n, causal);
    if (nk <= 0) {
        *lse_out = -INFINITY;
        return 0;
    }
    double mx = -INFINITY;
    for (long j = 0; j < nk; ++j) {
        const double *kj = kh + j * d;
        double s = 0.0;
        for (long t = 0; t < d; ++t) s += qi[t] * kj[t];
        s *= scale;
        p[j] = s;
        if (s > mx) mx = s;
    }
    double z = 0.0;
    for (long j = 0; j < nk; ++j) {
        p[j] = exp(p[j] - mx);
        z += p[j];
    }
    for (long j = 0; j < nk; ++j) p[j] /= z;
    *lse_out = mx + log(z);
    return nk;
}

/* O_i = sum_j P_ij V_j */
static void weighted_values(const double *p, long nk, const double *vh, long d, double *oi) {
    for (long t = 0; t < d; ++t) oi[t] = 0.0;
    for (long j = 0; j < nk; ++j) {
        const double *vj = vh + j * d;
        double pj = p[j];
        for (long t = 0; t < d; ++t) oi[t] += pj * vj[t];
    }
}

/*
 * Forward for the query rows listed in rows[0..nrows) of every head.
 * o: [B*H, nrows, d], lse: [B*H, nrows].  rows == NULL means every row
 * (nrows must then equal n).
 */
int oracle_fwd_rows(const double *q, const double *k, const double *v, long bh, long n,
                    long d, double scale, int causal, const long *rows, long nrows,
                    double *o, double *lse) {
    if (bh < 0 || n < 0 || d <= 0 || nrows < 0) return 1;
    if (rows == NULL && nrows != n) return 1;
    for (long r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= n) return 1;
    long total = bh * nrows;
    int failed = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        if (!p) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long idx = 0; idx < total; ++idx) {
            if (!p) continue;
            long h = idx / nrows, r = idx % nrows;
            long i = rows ? rows[r] : r;
            const double *qh = q + h * n * d, *kh = k + h * n * d, *vh = v + h * n * d;
            long nk = softmax_row(qh + i * d, kh, i, n, d, scale, causal, p, &lse[idx]);
            weighted_values(p, nk, vh, d, o + idx * d);
        }
        free(p);
    }
    return failed ? 2 : 0;
}

int oracle_fwd(const double *q, const double *k, const double *v, long bh, long n, long d,
               double scale, int causal, double *o, double *lse) {
    return oracle_fwd_rows(q, k, v, bh, n, d, scale, causal, NULL, n, o, lse);
}

/*
 * Backward restricted to the query rows rows[0..nrows) of every head (rows == NULL:
 * every row, nrows == n).  dq_rows [B*H, nrows, d] receives dQ of the listed rows;
 * dk and dv [B*H, n, d] receive the contributions of exactly the listed rows
 * (sum over i in rows of scale*dS_ij*Q_i and P_ij*dO_i).  With every row listed the
 * result is the full gradient of sum(O o dO) with respect to Q, K and V.  O and the
 * softmax are recomputed here from the definition.  Heads run in parallel; inside a
 * head the rows run in order, because dK and dV sum over rows.
 */
int oracle_bwd_rows(const double *q, const double *k, const double *v, const double *dout,
                    long bh, long n, long d, double scale, int causal, const long *rows,
                    long nrows, double *dq_rows, double *dk, double *dv) {
    if (bh < 0 || n < 0 || d <= 0 || nrows < 0) return 1;
    if (rows == NULL && nrows != n) return 1;
    for (long r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= n) return 1;
    int failed = 0;
#pragma omp parallel
    {
        size_t nn = (size_t)(n > 0 ? n : 1);
        double *p = (double *)malloc(sizeof(double) * nn);
        double *dp = (double *)malloc(sizeof(double) * nn);
        double *oi = (double *)malloc(sizeof(double) * (size_t)d);
        if (!p || !dp || !oi) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long h = 0; h < bh; ++h) {
            if (!p || !dp || !oi) continue;
            const double *qh = q + h * n * d, *kh = k + h * n * d, *vh = v + h * n * d;
            const double *doh = dout + h * n * d;
            double *dqh = dq_rows + h * nrows * d, *dkh = dk + h * n * d, *dvh = dv + h * n * d;
            memset(dkh, 0, sizeof(double) * (size_t)(n * d));
            memset(dvh, 0, sizeof(double) * (size_t)(n * d));
            for (long r = 0; r < nrows; ++r) {
                long i = rows ? rows[r] : r;
                const double *qi = qh + i * d, *doi = doh + i * d;
                double lse_i;
                long nk = softmax_row(qi, kh, i, n, d, scale, causal, p, &lse_i);
                weighted_values(p, nk, vh, d, oi);
                /* D_i = dO_i . O_i */
                double di = 0.0;
                for (long t = 0; t < d; ++t) di += doi[t] * oi[t];
                /* dP_ij = dO_i . V_j ;  dS_ij = P_ij (dP_ij - D_i) */
                for (long j = 0; j < nk; ++j) {
                    const double *vj = vh + j * d;
                    double s = 0.0;
                    for (long t = 0; t < d; ++t) s += doi[t] * vj[t];
                    dp[j] = p[j] * (s - di);
                }
                /* dQ_i = scale * sum_j dS_ij K_j */
                double *dqi = dqh + r * d;
                for (long t = 0; t < d; ++t) dqi[t] = 0.0;
                for (long j = 0; j < nk; ++j) {
                    const double *kj = kh + j * d;
                    for (long t = 0; t < d; ++t) dqi[t] += dp[j] * kj[t];
                }
                for (long t = 0; t < d; ++t) dqi[t] *= scale;
                /* dK_j += scale * dS_ij Q_i ;  dV_j += P_ij dO_i */
                for (long j = 0; j < nk; ++j) {
                    double *dkj = dkh + j * d, *dvj = dvh + j * d;
                    double a = scale * dp[j], b = p[j];
                    for (long t = 0; t < d; ++t) {
                        dkj[t] += a * qi[t];
                        dvj[t] += b * doi[t];
                    }
                }
            }
        }
        free(p);
        free(dp);
        free(oi);
    }
    return failed ? 2 : 0;
}

/* Backward for every head: the gradients of sum(O o dO) with respect to Q, K, V. */
int oracle_bwd(const double *q, const double *k, const double *v, const double *dout,
               long bh, long n, long d, double scale, int causal, double *dq, double *dk,
               double *dv) {
    return oracle_bwd_rows(q, k, v, dout, bh, n, d, scale, causal, NULL, n, dq, dk, dv);
}

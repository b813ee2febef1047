/*
 * Parallax forward oracle: a plain, slow, fp64 CPU implementation.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes (page "Parallax: parametrized local linear attention for
 * language modeling", section "Core mechanism" / "Kernmechanismus", the output
 * equation o^PLX_i = o^SA_i - Sigma_KV^(i) rho_i):
 *
 *   for one query i attending to keys j = 0 .. n-1
 *     s_j      = tau * <q_i, k_j>                       (softmax scores)
 *     w_j      = exp(s_j) / sum_l exp(s_l)               (softmax weights)
 *     o^SA     = sum_j w_j v_j                           (softmax attention)
 *     mu       = sum_j w_j k_j                           (weighted key mean)
 *     Sigma    = sum_j w_j (v_j - o^SA)(k_j - mu)^T      (d_v x d_k, formed
 *                                                         explicitly)
 *     o        = o^SA - Sigma rho_i
 *     lse      = log sum_j exp(s_j)
 *     cor      = |Sigma rho_i| / |o|                     (Euclidean norms;
 *                                                         0 when |o| = 0)
 *
 * The pages call Sigma_KV only "the KV covariance matrix"; the softmax-weighted
 * centred cross-covariance above is the reading used throughout this project.
 * cor is the correction-to-output ratio (COR) that the same page reports per
 * layer in its experimental results (optimizer dependence); the pages give no
 * formula, and the ratio of the Euclidean norms of the correction term and of
 * the output, per query, is the reading used here.
 * The steps are taken in the order of that definition, with no fusion: the
 * weights are normalised first, then the two weighted means, then the full
 * d x d matrix, then the matrix-vector product.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* One query against the first n rows of K and V (row-major, d doubles per
 * row, rows ks / vs doubles apart). Writes out[d] and *lse; if sigma_out is
 * not NULL it also receives the d x d matrix Sigma (row a = value dim,
 * column c = key dim), and if cor is not NULL the ratio |Sigma rho| / |o|.
 * Returns 0 on success, -1 on allocation failure.
 * n == 0 yields out = 0, lse = -inf and cor = 0. */
int plx_oracle_query(int n, int d, double tau,
                     const double *q, const double *rho,
                     const double *K, long ks, const double *V, long vs,
                     double *out, double *lse, double *sigma_out, double *cor)
{
    if (n <= 0) {
        for (int a = 0; a < d; ++a) out[a] = 0.0;
        *lse = -INFINITY;
        if (sigma_out) memset(sigma_out, 0, sizeof(double) * (size_t)d * d);
        if (cor) *cor = 0.0;
        return 0;
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    double *osa = (double *)calloc((size_t)d, sizeof(double));
    double *mu = (double *)calloc((size_t)d, sizeof(double));
    double *kc = (double *)malloc(sizeof(double) * (size_t)d);
    double *S = (double *)calloc((size_t)d * d, sizeof(double));
    if (!w || !osa || !mu || !kc || !S) {
        free(w); free(osa); free(mu); free(kc); free(S);
        return -1;
    }

    /* 1. scores and softmax weights (shifted by the maximum for range only) */
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        const double *kj = K + (long)j * ks;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += q[c] * kj[c];
        s *= tau;
        w[j] = s;
        if (s > m) m = s;
    }
    double Z = 0.0;
    for (int j = 0; j < n; ++j) {
        w[j] = exp(w[j] - m);
        Z += w[j];
    }
    for (int j = 0; j < n; ++j) w[j] /= Z;
    *lse = m + log(Z);

    /* 2. softmax attention output and weighted key mean */
    for (int j = 0; j < n; ++j) {
        const double *kj = K + (long)j * ks;
        const double *vj = V + (long)j * vs;
        for (int a = 0; a < d; ++a) {
            osa[a] += w[j] * vj[a];
            mu[a] += w[j] * kj[a];
        }
    }

    /* 3. the weighted, centred KV cross-covariance, explicitly */
    for (int j = 0; j < n; ++j) {
        const double *kj = K + (long)j * ks;
        const double *vj = V + (long)j * vs;
        for (int c = 0; c < d; ++c) kc[c] = kj[c] - mu[c];
        for (int a = 0; a < d; ++a) {
            const double coef = w[j] * (vj[a] - osa[a]);
            double *Sa = S + (size_t)a * d;
            for (int c = 0; c < d; ++c) Sa[c] += coef * kc[c];
        }
    }

    /* 4. o = o^SA - Sigma rho, and the norms of the correction and of o */
    double corr_sq = 0.0, out_sq = 0.0;
    for (int a = 0; a < d; ++a) {
        const double *Sa = S + (size_t)a * d;
        double corr = 0.0;
        for (int c = 0; c < d; ++c) corr += Sa[c] * rho[c];
        out[a] = osa[a] - corr;
        corr_sq += corr * corr;
        out_sq += out[a] * out[a];
    }
    if (cor) *cor = out_sq > 0.0 ? sqrt(corr_sq) / sqrt(out_sq) : 0.0;
    if (sigma_out) memcpy(sigma_out, S, sizeof(double) * (size_t)d * d);

    free(w); free(osa); free(mu); free(kc); free(S);
    return 0;
}

/* A batch of queries that share one key/value set: query r (row r of Q and R,
 * d doubles each) attends to the first nkeys[r] rows of K and V. Serves both
 * causal prefill (nkeys = i + 1) and decode (nkeys = cache length). cor may
 * be NULL; otherwise it receives one ratio per row. */
int plx_oracle_rows(int nrows, const int *nkeys, int d, double tau,
                    const double *Q, const double *R,
                    const double *K, const double *V,
                    double *out, double *lse, double *cor)
{
    for (int r = 0; r < nrows; ++r) {
        int rc = plx_oracle_query(nkeys[r], d, tau, Q + (size_t)r * d, R + (size_t)r * d,
                                  K, d, V, d, out + (size_t)r * d, lse + r, NULL,
                                  cor ? cor + r : NULL);
        if (rc) return rc;
    }
    return 0;
}

/*
 * aatc_oracle.c -- plain, slow, fp64 CPU reference for Attention-Aware
 * Transform Coding (AATC) of KV caches.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA path is
 * checked against.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load it; the product library never does, and the
 * two share no code, headers, tables or constants.
 *
 * Every function follows one step of the method as the pages describe it:
 *   [KLT]  "Attention-Aware Transform Coding Guide: KV Compression",
 *          section "Decorrelation via the Karhunen-Loeve Transform (KLT)".
 *   [RWF]  same page, section "Optimal Bit Allocation via Reverse
 *          Water-Filling".
 *   [ATT]  same page, section "Formal Attention Distortion Model".
 *   [THM]  same page, section "Theorem: Additive Error Decomposition".
 *   [IMPL] same page, section "End-to-End Implementation" (the PyTorch
 *          sketch: covariance, eigh, bisection water-filling, rotate and
 *          quantize per channel).
 *   [NOVA] "Spend Bits Where Queries Look: KV Cache Vector Quantization with
 *          Attention-Preserving Transforms", Abstract (non-orthogonal key
 *          transform, generalized Parseval relation, fixed per-token bit
 *          count, bandwidth-bound decoding).
 *
 * Readings taken where the pages are silent or disagree are stated at each
 * function.  Parity pins for every function live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_MAXB 8 /* largest per-channel bit width */

int orc_abi_version(void) { return 2; }

/* ------------------------------------------------------------------------ */
/* Statistics  [KLT], [IMPL] covariance step                                 */
/* ------------------------------------------------------------------------ */

/* mu[j] = (1/n) sum_i X[i][j].  X is [n][d] row-major. */
void orc_mean(const double *X, long n, int d, double *mu)
{
    for (int j = 0; j < d; ++j) mu[j] = 0.0;
    for (long i = 0; i < n; ++i)
        for (int j = 0; j < d; ++j) mu[j] += X[i * d + j];
    for (int j = 0; j < d; ++j) mu[j] /= (double)n;
}

/* S = (1/n) sum_i (x_i - c)(x_i - c)^T.
 * With c = mean this is the centered channel covariance of K or V (reading:
 * the sketch's torch.cov centers; the 1/n vs 1/(n-1) factor scales all
 * eigenvalues and steps together and leaves every code unchanged).
 * With c = NULL it is the uncentered second moment E[x x^T] that the
 * query metric needs ([THM]: key error enters through q . e with raw q). */
void orc_moment(const double *X, long n, int d, const double *c, double *S)
{
    double *row = (double *)malloc(sizeof(double) * d);
    for (int a = 0; a < d * d; ++a) S[a] = 0.0;
    for (long i = 0; i < n; ++i) {
        for (int j = 0; j < d; ++j) row[j] = X[i * d + j] - (c ? c[j] : 0.0);
        for (int a = 0; a < d; ++a)
            for (int b = 0; b < d; ++b) S[a * d + b] += row[a] * row[b];
    }
    for (int a = 0; a < d * d; ++a) S[a] /= (double)n;
    free(row);
}

/* ------------------------------------------------------------------------ */
/* Symmetric eigendecomposition by cyclic Jacobi  [KLT] Sigma = U Lambda U^T  */
/* ------------------------------------------------------------------------ */

/* Cyclic-by-row two-sided Jacobi (Golub & Van Loan, "Matrix Computations",
 * sec. 8.5).  A pair (p,q) is rotated unless |a_pq| <= tol*sqrt(|a_pp a_qq|);
 * the iteration stops after the first sweep in which no pair needed a
 * rotation.  On return evals are sorted in descending order (ties keep the
 * original index order) and column k of evecs ([d][d] row-major, element
 * [i][k]) is the unit eigenvector of evals[k], signed so that its entry of
 * largest magnitude (lowest index on ties) is positive.
 * Returns the number of sweeps used, or -1 if max_sweeps was not enough. */
int orc_jacobi_eig(const double *A_in, int d, int max_sweeps, double tol,
                   double *evals, double *evecs)
{
    double *A = (double *)malloc(sizeof(double) * d * d);
    double *V = (double *)malloc(sizeof(double) * d * d);
    memcpy(A, A_in, sizeof(double) * d * d);
    for (int i = 0; i < d; ++i)
        for (int k = 0; k < d; ++k) V[i * d + k] = (i == k) ? 1.0 : 0.0;

    int sweeps = 0, converged = 0;
    while (sweeps < max_sweeps) {
        int rotated = 0;
        for (int p = 0; p < d - 1; ++p) {
            for (int q = p + 1; q < d; ++q) {
                double apq = A[p * d + q];
                double app = A[p * d + p], aqq = A[q * d + q];
                if (fabs(apq) <= tol * sqrt(fabs(app * aqq))) continue;
                rotated = 1;
                /* symmetric 2x2 Schur decomposition */
                double tau = (aqq - app) / (2.0 * apq);
                double t = (tau >= 0.0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
                double c = 1.0 / sqrt(1.0 + t * t);
                double s = t * c;
                /* A <- J^T A J with J_pp = c, J_pq = s, J_qp = -s, J_qq = c */
                for (int k = 0; k < d; ++k) {
                    if (k == p || k == q) continue;
                    double akp = A[k * d + p], akq = A[k * d + q];
                    double nkp = c * akp - s * akq;
                    double nkq = s * akp + c * akq;
                    A[k * d + p] = nkp; A[p * d + k] = nkp;
                    A[k * d + q] = nkq; A[q * d + k] = nkq;
                }
                double npp = c * c * app - 2.0 * c * s * apq + s * s * aqq;
                double nqq = s * s * app + 2.0 * c * s * apq + c * c * aqq;
                A[p * d + p] = npp;
                A[q * d + q] = nqq;
                A[p * d + q] = 0.0;
                A[q * d + p] = 0.0;
                /* V <- V J */
                for (int k = 0; k < d; ++k) {
                    double vkp = V[k * d + p], vkq = V[k * d + q];
                    V[k * d + p] = c * vkp - s * vkq;
                    V[k * d + q] = s * vkp + c * vkq;
                }
            }
        }
        ++sweeps;
        if (!rotated) { converged = 1; break; }
    }

    /* sort descending, stable in the original index (insertion sort) */
    int *idx = (int *)malloc(sizeof(int) * d);
    for (int k = 0; k < d; ++k) idx[k] = k;
    for (int a = 1; a < d; ++a) {
        int key = idx[a];
        double kv = A[key * d + key];
        int b = a - 1;
        while (b >= 0 && A[idx[b] * d + idx[b]] < kv) { idx[b + 1] = idx[b]; --b; }
        idx[b + 1] = key;
    }
    for (int k = 0; k < d; ++k) {
        int src = idx[k];
        evals[k] = A[src * d + src];
        int arg = 0;
        double best = -1.0;
        for (int i = 0; i < d; ++i) {
            double m = fabs(V[i * d + src]);
            if (m > best) { best = m; arg = i; }
        }
        double sg = V[arg * d + src] < 0.0 ? -1.0 : 1.0;
        for (int i = 0; i < d; ++i) evecs[i * d + k] = sg * V[i * d + src];
    }
    free(idx); free(A); free(V);
    return converged ? sweeps : -1;
}

/* C = A * B for [d][d] matrices (row-major). */
static void matmul(const double *A, const double *B, double *C, int d)
{
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int k = 0; k < d; ++k) s += A[i * d + k] * B[k * d + j];
            C[i * d + j] = s;
        }
}

/* Key metric and KLT for one KV head.
 * [THM]: the key term of the distortion weights the key error by the query,
 * so the metric is the query second moment Sq = E[q q^T].  [NOVA]: the
 * optimal key transform is not orthogonal and turns the attention-aware key
 * distortion into plain MSE of the coefficients.  Reading: whiten by the
 * symmetric square root of Sq and then apply the KLT of the whitened key
 * covariance,
 *     M = Sq^{1/2} Sk Sq^{1/2} = Uk Lk Uk^T,
 *     Tk = Uk^T Sq^{1/2},   Tk^{-1} = Sq^{-1/2} Uk,   Ak = Tk^{-T} = Uk^T Sq^{-1/2}.
 * so that Tk^{-T} Sq Tk^{-1} = I and Tk Sk Tk^T = Lk.  Eigenvalues of Sq are
 * floored at 1e-12 of the largest before the inverse square root.
 * Outputs (all [d][d] row-major): Tk, Tk_inv, Ak, and the eigenvalues lamK.
 * Returns 0, or -1 if a Jacobi run did not converge. */
int orc_key_transform(const double *Sk, const double *Sq, int d, int max_sweeps,
                      double tol, double *Tk, double *Tk_inv, double *Ak,
                      double *lamK, double *lamQ)
{
    double *Uq = (double *)malloc(sizeof(double) * d * d);
    double *Sh = (double *)malloc(sizeof(double) * d * d);  /* Sq^{1/2}  */
    double *Si = (double *)malloc(sizeof(double) * d * d);  /* Sq^{-1/2} */
    double *M = (double *)malloc(sizeof(double) * d * d);
    double *tmp = (double *)malloc(sizeof(double) * d * d);
    double *Uk = (double *)malloc(sizeof(double) * d * d);
    int rc = 0;
    if (orc_jacobi_eig(Sq, d, max_sweeps, tol, lamQ, Uq) < 0) rc = -1;
    double floor_ = 1e-12 * (lamQ[0] > 0.0 ? lamQ[0] : 0.0);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            double sh = 0.0, si = 0.0;
            for (int k = 0; k < d; ++k) {
                double l = lamQ[k] > floor_ ? lamQ[k] : floor_;
                if (l <= 0.0) l = 1e-300;
                sh += Uq[i * d + k] * sqrt(l) * Uq[j * d + k];
                si += Uq[i * d + k] / sqrt(l) * Uq[j * d + k];
            }
            Sh[i * d + j] = sh;
            Si[i * d + j] = si;
        }
    matmul(Sh, Sk, tmp, d);
    matmul(tmp, Sh, M, d);
    for (int i = 0; i < d; ++i)          /* symmetrize rounding */
        for (int j = i + 1; j < d; ++j) {
            double a = 0.5 * (M[i * d + j] + M[j * d + i]);
            M[i * d + j] = a; M[j * d + i] = a;
        }
    if (orc_jacobi_eig(M, d, max_sweeps, tol, lamK, Uk) < 0) rc = -1;
    /* Tk = Uk^T Sh ; Ak = Uk^T Si ; Tk_inv = Si Uk */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            double t = 0.0, a = 0.0, v = 0.0;
            for (int k = 0; k < d; ++k) {
                t += Uk[k * d + i] * Sh[k * d + j];
                a += Uk[k * d + i] * Si[k * d + j];
                v += Si[i * d + k] * Uk[k * d + j];
            }
            Tk[i * d + j] = t;
            Ak[i * d + j] = a;
            Tk_inv[i * d + j] = v;
        }
    free(Uq); free(Sh); free(Si); free(M); free(tmp); free(Uk);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Reverse water-filling  [RWF]                                             */
/* ------------------------------------------------------------------------ */

/* Continuous solution: R_j = max(0, 1/2 log2(lam_j/theta)), D_j = min(theta,
 * lam_j), with sum_j R_j = total_bits (no upper clamp).  Solved exactly: for
 * an active set of the n largest eigenvalues, log2 theta = (sum_{j<n} log2
 * lam_j - 2 total)/n; the right n is the one with lam_{n-1} > theta >= lam_n.
 * lam must be sorted descending.  Returns theta. */
double orc_waterfill_theta(const double *lam, int d, double total_bits,
                           double *R, double *D)
{
    double slog = 0.0, theta = 0.0;
    for (int n = 1; n <= d; ++n) {
        if (!(lam[n - 1] > 0.0)) break;
        slog += log2(lam[n - 1]);
        double lt = (slog - 2.0 * total_bits) / n;
        double th = exp2(lt);
        double next = (n < d && lam[n] > 0.0) ? lam[n] : 0.0;
        theta = th;
        if (lam[n - 1] > th && th >= next) break;
    }
    for (int j = 0; j < d; ++j) {
        double l = lam[j] > 0.0 ? lam[j] : 0.0;
        R[j] = (l > theta) ? 0.5 * log2(l / theta) : 0.0;
        D[j] = l < theta ? l : theta;
    }
    return theta;
}

/* Integer allocation b_j in 0..8 with sum_j b_j = B_bits exactly.
 * The reduction of distortion from giving channel j its (t+1)-th bit is
 * proportional to the gain g_{j,t} = lam_j 4^{-t} (each bit quarters the
 * error variance at high resolution, [RWF]).  b_j is the number of gains of
 * channel j among the B_bits largest of all d*8 gains, ties going to the
 * smaller j and then the smaller t.  Because g_{j,t} falls strictly in t
 * this is the exact integer optimum of sum_j lam_j 4^{-b_j}.  Reading: the
 * pages give 0..8 ("pruned entirely (R_j = 0)") in one place and 2..8 in the
 * sketch; the range 0..8 is used.  Negative eigenvalues count as 0.
 * Also returns, in *margin, the relative gap between the B-th and (B+1)-th
 * largest gains (1.0 when there is no (B+1)-th). */
typedef struct { double g; int j, t; } gain_t;

static int gain_cmp(const void *a, const void *b)
{
    const gain_t *x = (const gain_t *)a, *y = (const gain_t *)b;
    if (x->g > y->g) return -1;
    if (x->g < y->g) return 1;
    if (x->j != y->j) return x->j < y->j ? -1 : 1;
    return x->t < y->t ? -1 : (x->t > y->t);
}

int orc_allocate_bits(const double *lam, int d, int B_bits, int *bits, double *margin)
{
    if (B_bits < 0 || B_bits > ORC_MAXB * d) return -1;
    int n = d * ORC_MAXB;
    gain_t *g = (gain_t *)malloc(sizeof(gain_t) * n);
    for (int j = 0; j < d; ++j)
        for (int t = 0; t < ORC_MAXB; ++t) {
            double l = lam[j] > 0.0 ? lam[j] : 0.0;
            g[j * ORC_MAXB + t].g = ldexp(l, -2 * t);
            g[j * ORC_MAXB + t].j = j;
            g[j * ORC_MAXB + t].t = t;
        }
    qsort(g, n, sizeof(gain_t), gain_cmp);
    for (int j = 0; j < d; ++j) bits[j] = 0;
    for (int k = 0; k < B_bits; ++k) bits[g[k].j] += 1;
    if (margin) {
        if (B_bits == 0 || B_bits >= n) *margin = 1.0;
        else {
            double a = g[B_bits - 1].g, b = g[B_bits].g;
            *margin = a > 0.0 ? (a - b) / a : 0.0;
        }
    }
    free(g);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Attention-aware token weights and the joint K/V budget split [THM], [RWF] */
/* ------------------------------------------------------------------------ */

/* [THM] writes the value distortion as sum_i A_i^2 sum_j sigma_Vij^2 and the
 * key distortion as (1/d) sum_j q_j^2 sum_i A_i^2 |v_i - o|^2 sigma_Kij^2.  A
 * fixed quantizer per channel gives every token the same noise variance, so
 * the token sums factor out of both:
 *   alpha_V = sum_i A_i^2,   alpha_K = (1/d) sum_i A_i^2 |v_i - o|^2.
 * Reading: both are averaged over m calibration queries Q [m][d], each of
 * which attends all n calibration keys K [n][d] (values V [n][d]) with the
 * 1/sqrt(d) scale and no mask.  The q_j^2 factor stays in the key metric (the
 * query second-moment whitening), so the per-channel key weights remain the
 * eigenvalues of the whitened key covariance.  Plain loops, exact softmax. */
void orc_attention_weights(const double *Q, const double *K, const double *V, long m, long n, int d,
                           double *alpha_k, double *alpha_v)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    const double scale = 1.0 / sqrt((double)d);
    double ak = 0.0, av = 0.0;
    for (long q = 0; q < m; ++q) {
        double mx = -INFINITY;
        for (long i = 0; i < n; ++i) {
            double dot = 0.0;
            for (int j = 0; j < d; ++j) dot += Q[q * d + j] * K[i * d + j];
            s[i] = dot * scale;
            if (s[i] > mx) mx = s[i];
        }
        double den = 0.0;
        for (long i = 0; i < n; ++i) {
            s[i] = exp(s[i] - mx);
            den += s[i];
        }
        for (int j = 0; j < d; ++j) o[j] = 0.0;
        double a2 = 0.0;
        for (long i = 0; i < n; ++i) {
            s[i] /= den; /* A_i */
            a2 += s[i] * s[i];
            for (int j = 0; j < d; ++j) o[j] += s[i] * V[i * d + j];
        }
        double r = 0.0;
        for (long i = 0; i < n; ++i) {
            double e2 = 0.0;
            for (int j = 0; j < d; ++j) {
                const double e = V[i * d + j] - o[j];
                e2 += e * e;
            }
            r += s[i] * s[i] * e2;
        }
        av += a2;
        ak += r / d;
    }
    free(s);
    free(o);
    *alpha_k = m > 0 ? ak / m : 0.0;
    *alpha_v = m > 0 ? av / m : 0.0;
}

/* Weighted high-rate distortion of an allocation: alpha sum_j lam_j 4^-b_j. */
static double alloc_cost(const double *lam, const int *bits, int d, double alpha)
{
    double c = 0.0;
    for (int j = 0; j < d; ++j) c += ldexp(lam[j] > 0.0 ? lam[j] : 0.0, -2 * bits[j]);
    return alpha * c;
}

/* [RWF] with the [THM] weights: one water level over the channels of K and V,
 * i.e. minimize sum_h alpha_Kh sum_j lam_Khj 4^-bKhj + alpha_Vh sum_j lam_Vhj 4^-bVhj
 * subject to sum_j bKhj + sum_j bVhj = B_total for each of the H heads of a
 * layer, 0 <= b <= 8.  Reading: a cache holds one record width per tensor for
 * every head of the layer, so the split B_K + B_V = B_total is common to the
 * heads and restricted to multiples of `granule` bits (32 for the record
 * format).  For each such split every head takes the exact top-B allocation of
 * each side (orc_allocate_bits), optimal for that budget; the split of least
 * total cost wins, ties going to the split nearest B_total / 2, then to the
 * smaller B_K.  lam_k, lam_v, bits_k, bits_v: [H][d].  Returns -1 for an
 * impossible budget. */
int orc_joint_allocation(const double *lam_k, const double *lam_v, int H, int d, const double *alpha_k,
                         const double *alpha_v, int B_total, int granule, int *bits_k, int *bits_v, int *B_k,
                         double *cost)
{
    if (H <= 0 || granule <= 0 || B_total < 0 || B_total > 2 * ORC_MAXB * d || B_total % granule) return -1;
    const size_t n = (size_t)H * d;
    int *tk = (int *)malloc(sizeof(int) * n), *tv = (int *)malloc(sizeof(int) * n);
    if (!tk || !tv) {
        free(tk);
        free(tv);
        return -1;
    }
    int best = -1;
    double best_cost = INFINITY;
    for (int bk = 0; bk <= B_total; bk += granule) {
        const int bv = B_total - bk;
        if (bk > ORC_MAXB * d || bv > ORC_MAXB * d) continue;
        double c = 0.0;
        for (int h = 0; h < H; ++h) {
            orc_allocate_bits(lam_k + (size_t)h * d, d, bk, tk + (size_t)h * d, NULL);
            orc_allocate_bits(lam_v + (size_t)h * d, d, bv, tv + (size_t)h * d, NULL);
            c += alloc_cost(lam_k + (size_t)h * d, tk + (size_t)h * d, d, alpha_k[h]) +
                 alloc_cost(lam_v + (size_t)h * d, tv + (size_t)h * d, d, alpha_v[h]);
        }
        const int better = best < 0 || c < best_cost ||
                           (c == best_cost && abs(2 * bk - B_total) < abs(2 * best - B_total));
        if (better) {
            best = bk;
            best_cost = c;
            memcpy(bits_k, tk, sizeof(int) * n);
            memcpy(bits_v, tv, sizeof(int) * n);
        }
    }
    free(tk);
    free(tv);
    if (best < 0) return -1;
    *B_k = best;
    *cost = best_cost;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step sizes: MSE-optimal uniform quantizer for a unit Gaussian            */
/* ------------------------------------------------------------------------ */

static double phi(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
static double Phi(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* MSE of a mid-rise uniform quantizer with N = 2^b levels y_u = (u-(N-1)/2)D
 * and thresholds halfway between levels, for x ~ N(0,1).  Exact integral:
 * int_a^b (x-y)^2 phi = [Phi]_a^b (1 + y^2) + (a - 2y) phi(a) - (b - 2y) phi(b). */
double orc_gauss_uniform_mse(int b, double D)
{
    long N = 1L << b;
    double mse = 0.0;
    for (long u = 0; u < N; ++u) {
        double y = ((double)u - 0.5 * (double)(N - 1)) * D;
        double lo = (u == 0) ? -INFINITY : ((double)u - 0.5 * (double)N) * D;
        double hi = (u == N - 1) ? INFINITY : ((double)u + 1.0 - 0.5 * (double)N) * D;
        double P = Phi(hi) - Phi(lo);
        double pa = isinf(lo) ? 0.0 : (lo - 2.0 * y) * phi(lo);
        double pb = isinf(hi) ? 0.0 : (hi - 2.0 * y) * phi(hi);
        mse += P * (1.0 + y * y) + pa - pb;
    }
    return mse;
}

/* d MSE / d D up to the factor 2/D: sum_u y_u (y_u P_u - m_u) with
 * m_u = int_cell x phi = phi(lo) - phi(hi).  (The moving thresholds add
 * nothing because they sit halfway between neighbouring levels.) */
static double mse_slope(int b, double D)
{
    long N = 1L << b;
    double f = 0.0;
    for (long u = 0; u < N; ++u) {
        double y = ((double)u - 0.5 * (double)(N - 1)) * D;
        double lo = (u == 0) ? -INFINITY : ((double)u - 0.5 * (double)N) * D;
        double hi = (u == N - 1) ? INFINITY : ((double)u + 1.0 - 0.5 * (double)N) * D;
        double P = Phi(hi) - Phi(lo);
        double m = (isinf(lo) ? 0.0 : phi(lo)) - (isinf(hi) ? 0.0 : phi(hi));
        f += y * (y * P - m);
    }
    return f;
}

/* The step s_b minimizing orc_gauss_uniform_mse(b, .).  Golden-section search
 * brackets the minimum of the exact MSE integral; bisection on the sign of
 * its derivative then resolves it to the last bit.  Reading: the pages scale
 * each channel by a dynamic max-abs over the sequence; a static per-channel
 * step from the calibration eigenvalue, Delta_j = s_b sqrt(lam_j) (Gaussian
 * high-resolution model of [THM] and [NOVA]), keeps the per-token record
 * fixed-width and needs no second pass over the cache. */
double orc_gauss_uniform_step(int b)
{
    if (b <= 0) return 0.0;
    const double gr = 0.5 * (sqrt(5.0) - 1.0);
    double a = 1e-4, c = 4.0;
    double x1 = c - gr * (c - a), x2 = a + gr * (c - a);
    double f1 = orc_gauss_uniform_mse(b, x1), f2 = orc_gauss_uniform_mse(b, x2);
    for (int it = 0; it < 200 && (c - a) > 1e-6; ++it) {
        if (f1 < f2) { c = x2; x2 = x1; f2 = f1; x1 = c - gr * (c - a); f1 = orc_gauss_uniform_mse(b, x1); }
        else         { a = x1; x1 = x2; f1 = f2; x2 = a + gr * (c - a); f2 = orc_gauss_uniform_mse(b, x2); }
    }
    double lo = a * 0.9, hi = c * 1.1;           /* slope < 0 at lo, > 0 at hi */
    for (int it = 0; it < 400; ++it) {
        double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (mse_slope(b, mid) < 0.0) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

/* Delta_j rounded to fp32 (the stored step), 0 for pruned channels. */
void orc_steps(const double *lam, const int *bits, int d, float *step)
{
    for (int j = 0; j < d; ++j) {
        if (bits[j] <= 0) { step[j] = 0.0f; continue; }
        double l = lam[j] > 0.0 ? lam[j] : 0.0;
        step[j] = (float)(orc_gauss_uniform_step(bits[j]) * sqrt(l));
    }
}

/* ------------------------------------------------------------------------ */
/* Quantize  [IMPL] per-channel rounding and clamping                        */
/* ------------------------------------------------------------------------ */

/* u_j = clamp(rint(v_j), 0, 2^b_j - 1) with v_j = c_j/Delta_j + (2^b_j-1)/2
 * rounded to fp32 before rint (round half to even).  Mid-rise levels are
 * symmetric about zero.  Reading: the sketch's mid-tread levels
 * +-(2^{b-1}-1) have no level at all for b = 1, so mid-rise is used.
 * u_j = 0 for pruned channels (b_j = 0), which decode to the mean. */
void orc_quantize(const double *c, const float *step, const int *bits, int d, int *u)
{
    for (int j = 0; j < d; ++j) {
        int b = bits[j];
        if (b <= 0) { u[j] = 0; continue; }
        double top = (double)((1 << b) - 1);
        float v = (float)(c[j] / (double)step[j] + 0.5 * top);
        double r = rint((double)v);
        if (r < 0.0) r = 0.0;
        if (r > top) r = top;
        u[j] = (int)r;
    }
}

/* pre-rounding value v_j (fp32) of orc_quantize, for tie analysis */
void orc_prequant(const double *c, const float *step, const int *bits, int d, float *v)
{
    for (int j = 0; j < d; ++j) {
        int b = bits[j];
        v[j] = b <= 0 ? 0.0f : (float)(c[j] / (double)step[j] + 0.5 * (double)((1 << b) - 1));
    }
}

/* c_hat_j = (u_j - (2^b_j-1)/2) Delta_j, 0 for pruned channels. */
void orc_dequantize(const int *u, const float *step, const int *bits, int d, double *c)
{
    for (int j = 0; j < d; ++j) {
        int b = bits[j];
        c[j] = b <= 0 ? 0.0 : ((double)u[j] - 0.5 * (double)((1 << b) - 1)) * (double)step[j];
    }
}

/* ------------------------------------------------------------------------ */
/* Fixed-width record layout  [NOVA] "fixed per-token bit count"            */
/* ------------------------------------------------------------------------ */

/* Reading (the pages fix only that every token takes the same number of
 * bits): a record of B = sum_j b_j bits, stored as B/32 little-endian u32
 * words, record bit k being bit k%32 of word k/32.  Each code u_j is stored
 * whole, in b_j consecutive record bits, least significant bit first.
 * Pruned channels (b_j = 0) take no bits.  The channels follow one another
 * in the order given by orc_record_order:
 *
 *   candidates = channels with b_j > 0;  p2 = p1 = 8;
 *   repeat until no candidate is left:
 *       need = 7 - p2 - p1;
 *       pick the candidate of smallest width b >= need (ties: smallest j);
 *       if no candidate is that wide, pick the widest (ties: smallest j);
 *       append it;  p2 = p1;  p1 = its width.
 *
 * The rule tries to keep any three consecutive codes at 7 bits or more, so
 * that few bytes of the record hold parts of more than four codes (the
 * decoder is fastest then; correctness does not depend on it: the layout is
 * defined by the rule above alone).
 * order[0..n-1] receives the channel order; returns n. */
int orc_record_order(const int *bits, int d, int *order)
{
    char *used = (char *)calloc((size_t)d, 1);
    int n = 0, total = 0, p2 = 8, p1 = 8;
    for (int j = 0; j < d; ++j) total += bits[j] > 0;
    while (n < total) {
        int need = 7 - p2 - p1, pick = -1, widest = -1;
        for (int j = 0; j < d; ++j) {
            if (used[j] || bits[j] <= 0) continue;
            if (bits[j] >= need && (pick < 0 || bits[j] < bits[pick])) pick = j;
            if (widest < 0 || bits[j] > bits[widest]) widest = j;
        }
        if (pick < 0) pick = widest;
        used[pick] = 1;
        order[n++] = pick;
        p2 = p1;
        p1 = bits[pick];
    }
    free(used);
    return n;
}

/* off[j] = record bit offset of the code of channel j, -1 if b_j = 0. */
void orc_layout(const int *bits, int d, int *off)
{
    int *order = (int *)malloc(sizeof(int) * (d > 0 ? d : 1));
    int n = orc_record_order(bits, d, order), pos = 0;
    for (int j = 0; j < d; ++j) off[j] = -1;
    for (int k = 0; k < n; ++k) { off[order[k]] = pos; pos += bits[order[k]]; }
    free(order);
}

void orc_pack(const int *u, const int *bits, int d, int W, uint32_t *rec)
{
    int *off = (int *)malloc(sizeof(int) * d);
    orc_layout(bits, d, off);
    for (int w = 0; w < W; ++w) rec[w] = 0u;
    for (int j = 0; j < d; ++j) {
        if (off[j] < 0) continue;
        for (int k = 0; k < bits[j]; ++k)       /* bit by bit: obviously right */
            if (((uint32_t)u[j] >> k) & 1u) rec[(off[j] + k) >> 5] |= 1u << ((off[j] + k) & 31);
    }
    free(off);
}

void orc_unpack(const uint32_t *rec, const int *bits, int d, int *u)
{
    int *off = (int *)malloc(sizeof(int) * d);
    orc_layout(bits, d, off);
    for (int j = 0; j < d; ++j) {
        uint32_t v = 0;
        if (off[j] >= 0)
            for (int k = 0; k < bits[j]; ++k)
                if ((rec[(off[j] + k) >> 5] >> ((off[j] + k) & 31)) & 1u) v |= 1u << k;
        u[j] = (int)v;
    }
    free(off);
}

/* ------------------------------------------------------------------------ */
/* Cache tiling: where each token's record lives in the packed cache        */
/* ------------------------------------------------------------------------ */

/* Reading (the pages give no cache layout): the cache of one (batch row,
 * KV head) is a run of 32-token tiles, tile t holding tokens 32t..32t+31 in
 * 32*W consecutive words.  Within a tile, token i (0..31):
 *
 * keys (kind 0): half h = i/16 covers words [16W h, 16W (h+1)); inside it
 *   record word w sits in row r = w/4 (rows of n_r = min(4, W-4r) words,
 *   row r starting 64 r words into the half), at
 *       64 r + (i%16 / 2) * 2 n_r + 2 (w - 4r) + (i % 2);
 *   i.e. for each row, token pairs in order, each pair giving its row words
 *   in order, the two tokens of a pair side by side.
 * values (kind 1): the record is read as 2W half-words (half-word e = bits
 *   16e..16e+15 of the record); word 16 e + i/2 of the tile holds half-word e
 *   of token i in bits 0..15 when i is even and in bits 16..31 when i is odd.
 *
 * Both place every bit of every record exactly once.  Returns the word index
 * within the tile (keys) or the word index with *half = 0/1 (values). */
static long key_word_pos(int i, int w, int W)
{
    int r = w / 4, nr = W - 4 * r < 4 ? W - 4 * r : 4, ii = i % 16;
    return (long)16 * W * (i / 16) + 64L * r + (ii / 2) * 2L * nr + 2L * (w - 4 * r) + (ii % 2);
}

/* Write the records rec[n][W] of tokens start..start+n-1 into the cache
 * slab (words of tokens outside that range are left as they are). */
void orc_cache_put(const uint32_t *rec, long n, int W, int kind, long start, uint32_t *cache)
{
    for (long a = 0; a < n; ++a) {
        long t = start + a, base = (t / 32) * 32L * W;
        int i = (int)(t % 32);
        if (kind == 0) {
            for (int w = 0; w < W; ++w) cache[base + key_word_pos(i, w, W)] = rec[a * W + w];
        } else {
            for (int e = 0; e < 2 * W; ++e) {
                uint32_t hw = (rec[a * W + e / 2] >> (16 * (e % 2))) & 0xFFFFu;
                uint32_t *p = &cache[base + 16L * e + i / 2];
                if (i % 2) *p = (*p & 0x0000FFFFu) | (hw << 16);
                else       *p = (*p & 0xFFFF0000u) | hw;
            }
        }
    }
}

/* Read back the records of tokens start..start+n-1 from the cache slab. */
void orc_cache_get(const uint32_t *cache, long n, int W, int kind, long start, uint32_t *rec)
{
    for (long a = 0; a < n; ++a) {
        long t = start + a, base = (t / 32) * 32L * W;
        int i = (int)(t % 32);
        if (kind == 0) {
            for (int w = 0; w < W; ++w) rec[a * W + w] = cache[base + key_word_pos(i, w, W)];
        } else {
            for (int w = 0; w < W; ++w) rec[a * W + w] = 0u;
            for (int e = 0; e < 2 * W; ++e) {
                uint32_t hw = (cache[base + 16L * e + i / 2] >> (16 * (i % 2))) & 0xFFFFu;
                rec[a * W + e / 2] |= hw << (16 * (e % 2));
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Encode: transform, quantize, pack  ([KLT] K' = K U, [IMPL] compress)      */
/* ------------------------------------------------------------------------ */

/* For each of the n rows x of X ([n][d]):  c = T (x - mu), codes by
 * orc_quantize, record by orc_pack into rec[n][W].  If codes != NULL the
 * integer codes are also written ([n][d]); if pre != NULL the fp32
 * pre-rounding values are written ([n][d]). */
void orc_encode(const double *X, long n, int d, const double *T, const double *mu,
                const float *step, const int *bits, int W, uint32_t *rec,
                int *codes, float *pre)
{
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) {
        double *c = (double *)malloc(sizeof(double) * d);
        int *u = (int *)malloc(sizeof(int) * d);
        for (int a = 0; a < d; ++a) {
            double s = 0.0;
            for (int b = 0; b < d; ++b) s += T[a * d + b] * (X[i * d + b] - mu[b]);
            c[a] = s;
        }
        orc_quantize(c, step, bits, d, u);
        if (pre) orc_prequant(c, step, bits, d, pre + i * d);
        orc_pack(u, bits, d, W, rec + i * W);
        if (codes) for (int a = 0; a < d; ++a) codes[i * d + a] = u[a];
        free(c); free(u);
    }
}

/* ------------------------------------------------------------------------ */
/* Attention  [ATT]  o = softmax(q K^T / sqrt(d)) V                          */
/* ------------------------------------------------------------------------ */

/* Exact softmax attention of one query over L keys/values ([L][d]), with the
 * maximum logit subtracted before exponentiation.  No causal mask: a decode
 * query sees every cached token.  L = 0 gives o = 0. */
void orc_attention(const double *q, const double *K, const double *V, long L, int d,
                   double *o)
{
    for (int j = 0; j < d; ++j) o[j] = 0.0;
    if (L <= 0) return;
    double *s = (double *)malloc(sizeof(double) * L);
    double m = -INFINITY, scale = 1.0 / sqrt((double)d);
    for (long i = 0; i < L; ++i) {
        double a = 0.0;
        for (int j = 0; j < d; ++j) a += q[j] * K[i * d + j];
        s[i] = a * scale;
        if (s[i] > m) m = s[i];
    }
    double l = 0.0;
    for (long i = 0; i < L; ++i) { s[i] = exp(s[i] - m); l += s[i]; }
    for (long i = 0; i < L; ++i)
        for (int j = 0; j < d; ++j) o[j] += s[i] * V[i * d + j];
    for (int j = 0; j < d; ++j) o[j] /= l;
    free(s);
}

/* Reconstruct rows from records: x_hat = Tinv c_hat + mu  (the sketch's
 * dequantize-then-inverse-rotate), rec [n][W] -> Xh [n][d]. */
void orc_reconstruct(const uint32_t *rec, long n, int d, int W, const double *Tinv,
                     const double *mu, const float *step, const int *bits, double *Xh)
{
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) {
        int *u = (int *)malloc(sizeof(int) * d);
        double *c = (double *)malloc(sizeof(double) * d);
        orc_unpack(rec + i * W, bits, d, u);
        orc_dequantize(u, step, bits, d, c);
        for (int a = 0; a < d; ++a) {
            double s = mu[a];
            for (int b = 0; b < d; ++b) s += Tinv[a * d + b] * c[b];
            Xh[i * d + a] = s;
        }
        free(u); free(c);
    }
    (void)W;
}

/* Decode attention over a packed cache for one batch row and all query heads
 * of one KV head: the G queries q [G][d] attend to the L reconstructed
 * tokens (keys via Tk_inv, values via Uv) -> out [G][d]. */
void orc_decode_head(const double *q, int G, const uint32_t *krec, const uint32_t *vrec,
                     long L, int d, int Wk, int Wv,
                     const double *Tk_inv, const double *mu_k, const float *step_k, const int *bits_k,
                     const double *Uv, const double *mu_v, const float *step_v, const int *bits_v,
                     double *out)
{
    double *Kh = (double *)malloc(sizeof(double) * (L > 0 ? L : 1) * d);
    double *Vh = (double *)malloc(sizeof(double) * (L > 0 ? L : 1) * d);
    if (L > 0) {
        orc_reconstruct(krec, L, d, Wk, Tk_inv, mu_k, step_k, bits_k, Kh);
        orc_reconstruct(vrec, L, d, Wv, Uv, mu_v, step_v, bits_v, Vh);
    }
#pragma omp parallel for schedule(static)
    for (int g = 0; g < G; ++g) orc_attention(q + g * d, Kh, Vh, L, d, out + g * d);
    free(Kh); free(Vh);
}

/* orc_unpack for n records rec [n][W] -> u [n][d] (test convenience). */
void orc_unpack_rows(const uint32_t *rec, long n, int W, const int *bits, int d, int *u)
{
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) orc_unpack(rec + i * W, bits, d, u + i * d);
}

// calib.cu -- device calibration pipeline: statistics, Jacobi eigensolver,
// whitened key transform, bit allocation, step sizes and codec tables.
//
// Follows "Attention-Aware Transform Coding Guide: KV Compression" sections
// "Decorrelation via the Karhunen-Loeve Transform (KLT)" (covariance + eigh)
// and "Optimal Bit Allocation via Reverse Water-Filling", with the key metric
// of "Theorem: Additive Error Decomposition" (key error weighted by the query)
// and the non-orthogonal key transform of "Spend Bits Where Queries Look",
// Abstract (generalized Parseval relation).
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace {

constexpr int D = AATC_D;
constexpr int MOMENT_CHUNK = 512;    // calibration rows per partial-moment block
constexpr double JACOBI_TOL = 1e-15; // rotate (p,q) unless |a_pq| <= tol sqrt(|a_pp a_qq|)

__device__ __forceinline__ double to_f64(float x) { return (double)x; }
__device__ __forceinline__ double to_f64(__nv_bfloat16 x) { return (double)__bfloat162float(x); }

// ---------------------------------------------------------------------------
// Statistics
// ---------------------------------------------------------------------------

// mu[m][j] = mean over the n rows of matrix m (X: [M][n][D]).  One block per
// matrix, one thread per channel, fp64 accumulation in row order.
template <typename T>
__global__ void k_mean(const T *__restrict__ X, long n, double *__restrict__ mu, uint32_t *status)
{
    const int m = blockIdx.x, j = threadIdx.x;
    const T *x = X + (size_t)m * n * D + j;
    double s = 0.0;
    bool bad = false;
    for (long i = 0; i < n; ++i) {
        double v = to_f64(x[i * D]);
        bad |= !isfinite(v);
        s += v;
    }
    mu[m * D + j] = s / (double)n;
    if (__syncthreads_or(bad) && j == 0) atomicOr(status, AATC_DEV_NONFINITE);
}

template <typename T>
__global__ void k_check_finite(const T *__restrict__ x, size_t n, uint32_t *status)
{
    bool bad = false;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        bad |= !isfinite(to_f64(x[i]));
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, AATC_DEV_NONFINITE);
}

// Partial sums of (x - c)(x - c)^T over one chunk of MOMENT_CHUNK rows of
// matrix m (blockIdx.y).  256 threads; thread (ty, tx) owns the 8x8 output
// tile rows 8ty.., cols 8tx..; rows are staged 32 at a time in shared memory
// as fp64 after subtracting the center.  partial: [M][nchunks][D][D].
template <typename T>
__global__ void __launch_bounds__(256) k_moment_partial(const T *__restrict__ X, long n,
                                                        const double *__restrict__ center,
                                                        double *__restrict__ partial)
{
    __shared__ double xs[32][D];
    const int m = blockIdx.y, chunk = blockIdx.x, nchunks = gridDim.x;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const T *x = X + (size_t)m * n * D;
    const long r0 = (long)chunk * MOMENT_CHUNK;
    const long r1 = min(n, r0 + MOMENT_CHUNK);
    double acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.0;
    for (long r = r0; r < r1; r += 32) {
        const int rows = (int)min((long)32, r1 - r);
        __syncthreads();
        for (int e = tid; e < 32 * D; e += 256) {
            int i = e / D, j = e % D;
            double v = 0.0;
            if (i < rows) v = to_f64(x[(r + i) * D + j]) - (center ? center[m * D + j] : 0.0);
            xs[i][j] = v;
        }
        __syncthreads();
        for (int i = 0; i < rows; ++i) {
            double a[8], b[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) { a[k] = xs[i][ty * 8 + k]; b[k] = xs[i][tx * 8 + k]; }
#pragma unroll
            for (int p = 0; p < 8; ++p)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[p][q] = fma(a[p], b[q], acc[p][q]);
        }
    }
    double *out = partial + ((size_t)m * nchunks + chunk) * D * D;
#pragma unroll
    for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) out[(ty * 8 + p) * D + tx * 8 + q] = acc[p][q];
}

// out[m] = (1/n) sum over chunks (in order) of partial[m][chunk].
__global__ void k_moment_reduce(const double *__restrict__ partial, int nchunks, long n,
                                double *__restrict__ out)
{
    const int m = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= D * D) return;
    const double *p = partial + (size_t)m * nchunks * D * D + e;
    double s = 0.0;
    for (int c = 0; c < nchunks; ++c) s += p[(size_t)c * D * D];
    out[(size_t)m * D * D + e] = s / (double)n;
}

// ---------------------------------------------------------------------------
// One-block parallel cyclic Jacobi for a symmetric 128x128 fp64 matrix.
// ---------------------------------------------------------------------------
// Shared memory: the upper triangle of A packed row-wise (8256 doubles) and
// the full accumulated rotation V (16384 doubles) = 197,120 bytes.  Each sweep
// runs the 127 rounds of a round-robin tournament: in round r index 127 meets
// r and (r+k) meets (r-k) mod 127 for k = 1..63, so every round applies 64
// disjoint plane rotations at once and a sweep meets every pair once.  The
// rotation for a pair is the symmetric 2x2 Schur decomposition (Golub & Van
// Loan, sec. 8.5); a pair is skipped when |a_pq| <= tol sqrt(|a_pp a_qq|), and
// the iteration stops after a sweep with no rotation (the same test as a
// cyclic-by-row order; only the order of rotations differs).
// Output: eigenvalues descending (ties by index), eigenvectors as columns of
// evecs [D][D], each signed so its largest-magnitude entry (lowest index on
// ties) is positive.  A sweep cap bounds the work; hitting it sets
// AATC_DEV_NO_CONVERGENCE.
constexpr int JAC_THREADS = 512;
constexpr int TRI = D * (D + 1) / 2;
constexpr int JAC_BLOCKS = 64 * 65 / 2;   // 2x2 blocks (pair k1 <= pair k2) of one round
constexpr int PRE_SWEEPS = 10;            // cap of the fp32 preconditioning sweeps
template <typename R>
constexpr size_t jac_smem()
{
    return (size_t)(TRI + D * D) * sizeof(R) + 64 * 2 * sizeof(R) + 64 * 2 * sizeof(int) + 4 * sizeof(int) +
           (size_t)JAC_BLOCKS * 2 * sizeof(uint16_t);
}

__device__ __forceinline__ int tri(int i, int j)
{
    if (i > j) { int t = i; i = j; j = t; }
    return i * D - (i * (i - 1)) / 2 + (j - i);
}

// Mixed precision: FP64 runs at a small fraction of the FP32 rate on this GPU,
// so the sweeps are split in two.  PRE (R = float) runs fp32 sweeps from the
// identity until the off-diagonal reaches fp32 rounding (a pair is skipped when
// |a_pq| <= 1e-6 sqrt(|a_pp a_qq|) or below 2^-23 of the largest diagonal
// entry) and writes the accumulated rotations V as fp64.  The host makes V
// orthogonal to fp64 precision (Newton-Schulz) and forms A' = V^T A V in fp64.
// The final pass (R = double) then runs the sweeps above on A', starting its
// accumulation from that V, so its output is the decomposition of A; it
// needs a few sweeps (quadratic convergence from the fp32 level) instead of
// about twelve.
//
// Two independent batches in one launch: blocks m < M0 take (Ain0, evals0,
// evecs0, V00)[m], the others (Ain1, evals1, evecs1, V01)[m - M0].  V0 NULL:
// start from the identity.  PRE writes only evecs (the raw rotations).
template <typename R, bool PRE>
__global__ void __launch_bounds__(JAC_THREADS) k_jacobi(const double *__restrict__ Ain0, double *__restrict__ evals0,
                                                        double *__restrict__ evecs0, const double *__restrict__ V00,
                                                        int M0, const double *__restrict__ Ain1,
                                                        double *__restrict__ evals1, double *__restrict__ evecs1,
                                                        const double *__restrict__ V01, int max_sweeps,
                                                        uint32_t *status)
{
    extern __shared__ __align__(16) unsigned char jsm[];
    R *A = reinterpret_cast<R *>(jsm);     // packed upper triangle
    R *V = A + TRI;                        // [D][D]
    R *cs = V + D * D;                     // [64][2]
    int *pq = (int *)(cs + 128);           // [64][2]
    int *flag = pq + 128;                  // [0] rotated, [1] nonfinite
    uint16_t *kpair = reinterpret_cast<uint16_t *>(flag + 4);   // [JAC_BLOCKS][2]: block -> (k1, k2)
    __shared__ R floor_s;
    const int tid = threadIdx.x;
    const bool second = (int)blockIdx.x >= M0;
    const int m = second ? blockIdx.x - M0 : blockIdx.x;
    const double *Ain = second ? Ain1 : Ain0;
    double *evals = second ? evals1 : evals0;
    double *evecs = second ? evecs1 : evecs0;
    const double *V0 = second ? V01 : V00;
    const double *Am = Ain + (size_t)m * D * D;
    for (int blk = tid; blk < JAC_BLOCKS; blk += JAC_THREADS) {
        int k2 = (int)((sqrt(8.0 * blk + 1.0) - 1.0) * 0.5);
        while (k2 * (k2 + 1) / 2 > blk) --k2;
        while ((k2 + 1) * (k2 + 2) / 2 <= blk) ++k2;
        kpair[2 * blk] = (uint16_t)(blk - k2 * (k2 + 1) / 2);
        kpair[2 * blk + 1] = (uint16_t)k2;
    }

    if (tid < 2) flag[tid] = 0;
    __syncthreads();
    for (int e = tid; e < D * D; e += JAC_THREADS) {
        int i = e / D, j = e % D;
        V[e] = V0 ? (R)V0[(size_t)m * D * D + e] : (R)((i == j) ? 1.0 : 0.0);
        if (i <= j) {
            double a = 0.5 * (Am[i * D + j] + Am[j * D + i]);
            if (!isfinite(a)) flag[1] = 1;
            A[tri(i, j)] = (R)a;
        }
    }
    __syncthreads();
    if (flag[1]) {
        if (tid == 0) atomicOr(status, AATC_DEV_NONFINITE);
        for (int e = tid; e < D * D; e += JAC_THREADS) evecs[(size_t)m * D * D + e] = 0.0;
        if (!PRE && tid < D) evals[m * D + tid] = 0.0;
        return;
    }
    if (PRE && tid == 0) {   // fp32 noise level: 2^-23 of the largest diagonal entry
        R mx = 0;
        for (int i = 0; i < D; ++i) mx = fmax(mx, fabs(A[tri(i, i)]));
        floor_s = mx * (R)1.1920929e-7;
    }

    const R tol = PRE ? (R)1e-6 : (R)JACOBI_TOL;
    const int sweeps_cap = PRE ? PRE_SWEEPS : max_sweeps;
    bool converged = false;
    for (int sweep = 0; sweep < sweeps_cap && !converged; ++sweep) {
        if (tid == 0) flag[0] = 0;
        __syncthreads();
        for (int r = 0; r < D - 1; ++r) {
            if (tid < 64) {
                int a, b;
                if (tid == 0) { a = r; b = D - 1; }
                else { a = (r + tid) % (D - 1); b = (r - tid + (D - 1)) % (D - 1); }
                int p = min(a, b), q = max(a, b);
                R apq = A[tri(p, q)], app = A[tri(p, p)], aqq = A[tri(q, q)];
                R c = 1, sn = 0;
                if (fabs(apq) > tol * sqrt(fabs(app * aqq)) && (!PRE || fabs(apq) > floor_s)) {
                    R tau = (aqq - app) / (2 * apq);
                    R t = (tau >= 0 ? (R)1 : (R)-1) / (fabs(tau) + sqrt(1 + tau * tau));
                    c = 1 / sqrt(1 + t * t);
                    sn = t * c;
                    flag[0] = 1;
                }
                pq[2 * tid] = p; pq[2 * tid + 1] = q;
                cs[2 * tid] = c; cs[2 * tid + 1] = sn;
            }
            __syncthreads();
            // A <- J^T A J, one 2x2 block (pair k1, pair k2) per task, k1 <= k2
            for (int blk = tid; blk < JAC_BLOCKS; blk += JAC_THREADS) {
                const int k1 = kpair[2 * blk], k2 = kpair[2 * blk + 1];
                int p1 = pq[2 * k1], q1 = pq[2 * k1 + 1];
                R c1 = cs[2 * k1], s1 = cs[2 * k1 + 1];
                if (k1 == k2) {
                    R app = A[tri(p1, p1)], aqq = A[tri(q1, q1)], apq = A[tri(p1, q1)];
                    if (s1 != 0) {
                        A[tri(p1, p1)] = c1 * c1 * app - 2 * c1 * s1 * apq + s1 * s1 * aqq;
                        A[tri(q1, q1)] = s1 * s1 * app + 2 * c1 * s1 * apq + c1 * c1 * aqq;
                        A[tri(p1, q1)] = 0;
                    }
                } else {
                    R c2 = cs[2 * k2], s2 = cs[2 * k2 + 1];
                    if (s1 == 0 && s2 == 0) continue;   // identity on this block (exactly)
                    int p2 = pq[2 * k2], q2 = pq[2 * k2 + 1];
                    int i_pp = tri(p1, p2), i_pq = tri(p1, q2), i_qp = tri(q1, p2), i_qq = tri(q1, q2);
                    R xpp = A[i_pp], xpq = A[i_pq], xqp = A[i_qp], xqq = A[i_qq];
                    // rows: R1^T X  (R = [[c, s], [-s, c]])
                    R ypp = c1 * xpp - s1 * xqp, ypq = c1 * xpq - s1 * xqq;
                    R yqp = s1 * xpp + c1 * xqp, yqq = s1 * xpq + c1 * xqq;
                    // columns: (R1^T X) R2
                    A[i_pp] = c2 * ypp - s2 * ypq;
                    A[i_pq] = s2 * ypp + c2 * ypq;
                    A[i_qp] = c2 * yqp - s2 * yqq;
                    A[i_qq] = s2 * yqp + c2 * yqq;
                }
            }
            // V <- V J
            for (int e = tid; e < D * 64; e += JAC_THREADS) {
                int i = e >> 6, k = e & 63;
                R c = cs[2 * k], sn = cs[2 * k + 1];
                if (sn == 0) continue;
                int p = pq[2 * k], q = pq[2 * k + 1];
                R vp = V[i * D + p], vq = V[i * D + q];
                V[i * D + p] = c * vp - sn * vq;
                V[i * D + q] = sn * vp + c * vq;
            }
            __syncthreads();
        }
        converged = (flag[0] == 0);
        __syncthreads();
    }
    if (PRE) {   // the raw rotations, for the fp64 pass
        for (int e = tid; e < D * D; e += JAC_THREADS) evecs[(size_t)m * D * D + e] = (double)V[e];
        return;
    }
    if (!converged && tid == 0) atomicOr(status, AATC_DEV_NO_CONVERGENCE);

    // sort descending (stable in index) and sign-normalize
    if (tid < D) {
        double li = A[tri(tid, tid)];
        int rank = 0;
        for (int k = 0; k < D; ++k) {
            double lk = A[tri(k, k)];
            rank += (lk > li) || (lk == li && k < tid);
        }
        evals[m * D + rank] = li;
        int arg = 0;
        double best = -1.0;
        for (int i = 0; i < D; ++i) {
            double v = fabs(V[i * D + tid]);
            if (v > best) { best = v; arg = i; }
        }
        double sg = V[arg * D + tid] < 0.0 ? -1.0 : 1.0;
        double *out = evecs + (size_t)m * D * D;
        for (int i = 0; i < D; ++i) out[i * D + rank] = sg * V[i * D + tid];
    }
}

// Q <- 1.5 Q - 0.5 Y (Y = Q Q^T Q): one Newton-Schulz step towards the
// orthogonal factor of Q, [M][D][D].
__global__ void k_ns_step(double *__restrict__ Q, const double *__restrict__ Y, size_t n)
{
    const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e < n) Q[e] = 1.5 * Q[e] - 0.5 * Y[e];
}

// ---------------------------------------------------------------------------
// Small fp64 products: C[m] = op(A[m]) diag(f(lam[m])) op(B[m])
// ---------------------------------------------------------------------------
enum DiagMode { DIAG_NONE = 0, DIAG_SQRT = 1, DIAG_INVSQRT = 2 };

// f(l) = sqrt / 1/sqrt of max(l, 1e-12 * lam[0]) (lam sorted descending).
__global__ void k_gemm64(const double *__restrict__ A, int transA, const double *__restrict__ lam,
                         int mode, const double *__restrict__ B, int transB, double *__restrict__ C)
{
    __shared__ double f[D];
    const int m = blockIdx.y;
    const double *Am = A + (size_t)m * D * D, *Bm = B + (size_t)m * D * D;
    if (threadIdx.x < D) {
        double v = 1.0;
        if (mode != DIAG_NONE) {
            double fl = 1e-12 * fmax(lam[m * D], 0.0);
            double l = fmax(lam[m * D + threadIdx.x], fl);
            if (l <= 0.0) l = 1e-300;
            v = (mode == DIAG_SQRT) ? sqrt(l) : 1.0 / sqrt(l);
        }
        f[threadIdx.x] = v;
    }
    __syncthreads();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= D * D) return;
    const int i = e / D, j = e % D;
    double s = 0.0;
    for (int k = 0; k < D; ++k) {
        double a = transA ? Am[k * D + i] : Am[i * D + k];
        double b = transB ? Bm[j * D + k] : Bm[k * D + j];
        s += a * f[k] * b;
    }
    C[(size_t)m * D * D + e] = s;
}

// Y[m] = X[m]^T for [M][D][D] fp64 matrices.
__global__ void k_transpose64(const double *__restrict__ X, double *__restrict__ Y)
{
    const int m = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= D * D) return;
    const int i = e / D, j = e % D;
    Y[(size_t)m * D * D + e] = X[(size_t)m * D * D + j * D + i];
}

// ---------------------------------------------------------------------------
// Bit allocation and step sizes
// ---------------------------------------------------------------------------

// The step sizes depend only on the width b: computed once on the host.
double gauss_pdf(double x) { return exp(-0.5 * x * x) * 0.3989422804014327; }
double gauss_cdf(double x) { return 0.5 * erfc(-x * 0.7071067811865476); }

// Centroid map of a mid-rise uniform quantizer with N levels on N(0,1): given
// the step D (which fixes the cells), the step whose levels c_u D best fit
// the cell means in the MSE sense, sum_u c_u E[x; cell_u] / sum_u c_u^2 P_u.
double centroid_step(int N, double Dlt)
{
    double num = 0.0, den = 0.0;
    for (int u = 0; u < N; ++u) {
        double c = u - 0.5 * (N - 1);
        double lo = (u - 0.5 * N) * Dlt, hi = (u + 1 - 0.5 * N) * Dlt;
        double Plo = (u == 0) ? 0.0 : gauss_cdf(lo), Phi = (u == N - 1) ? 1.0 : gauss_cdf(hi);
        double flo = (u == 0) ? 0.0 : gauss_pdf(lo), fhi = (u == N - 1) ? 0.0 : gauss_pdf(hi);
        num += c * (flo - fhi);
        den += c * c * (Phi - Plo);
    }
    return num / den;
}

// The MSE-optimal step is the fixed point of centroid_step; solved by the
// secant method on centroid_step(D) - D from D0 = 4/N.
double gauss_uniform_step(int b)
{
    const int N = 1 << b;
    double x0 = 4.0 / N, x1 = centroid_step(N, x0);
    double r0 = x1 - x0;
    for (int it = 0; it < 200; ++it) {
        double r1 = centroid_step(N, x1) - x1;
        if (r1 == 0.0 || r1 == r0) break;
        double x2 = x1 - r1 * (x1 - x0) / (r1 - r0);
        x0 = x1; r0 = r1; x1 = x2;
        if (fabs(x1 - x0) <= 1e-16 * x1) break;
    }
    return x1;
}

// One block of 1024 threads per (head, tensor); thread t owns the gain of
// channel j = t/8 for its (t%8+1)-th bit, g = lam_j 4^{-(t%8)}.  The B
// largest gains are selected exactly: a bisection over the ordered bit
// patterns of the non-negative doubles finds the B-th largest gain value g*
// (count(g >= lo) >= B > count(g >= hi) is kept invariant), every gain above
// g* is taken, and gains equal to g* are taken in (j, t) order until the
// budget is met.  b_j = number of taken gains of channel j.
// Delta_j = s_{b_j} sqrt(lam_j) rounded to fp32.
struct StepTable {
    double s[AATC_MAXB + 1];   // s[b] = MSE-optimal uniform step of N(0,1) at b bits, s[0] = 0
};

const StepTable &step_table()
{
    static const StepTable t = [] {
        StepTable r;
        r.s[0] = 0.0;
        for (int b = 1; b <= AATC_MAXB; ++b) r.s[b] = gauss_uniform_step(b);
        return r;
    }();
    return t;
}

// Exact top-B selection for one (head, tensor) by one block of 1024 threads;
// thread t owns gain g = lam_j 4^{-(t%8)} of channel j = t/8 and ends with
// nb[j] = b_j.  Every thread returns its gain.
__device__ double topB_alloc(const double *lam, int B, double *gain, int *nb, unsigned long long *mx)
{
    const int t = threadIdx.x;
    const int j = t >> 3, tb = t & 7;
    const double g = ldexp(fmax(lam[j], 0.0), -2 * tb);
    gain[t] = g;
    if (t < D) nb[t] = 0;
    if (t == 0) *mx = 0ull;
    __syncthreads();
    atomicMax(mx, (unsigned long long)__double_as_longlong(g));
    __syncthreads();
    long long lo = 0, hi = (long long)*mx + 1;   // count(g >= 0) = all >= B > 0 = count(g >= hi)
    while (hi - lo > 1) {
        long long mid = lo + (hi - lo) / 2;
        int c = __syncthreads_count(g >= __longlong_as_double(mid));
        if (c >= B) lo = mid; else hi = mid;
    }
    const double gstar = __longlong_as_double(lo);
    const int above = __syncthreads_count(g > gstar);
    bool take = g > gstar;
    if (g == gstar) {
        int before = 0;
        for (int k = 0; k < t; ++k) before += (gain[k] == gstar);
        take = (above + before) < B;
    }
    if (take) atomicAdd(&nb[j], 1);
    __syncthreads();
    return g;
}

// Budget B (0 < B <= 8 D) of tensor `tensor` (0 = keys): from the joint split
// chosen on the device when given, else the handle's own.
__global__ void __launch_bounds__(1024) k_waterfill(const double *__restrict__ lam_k,
                                                    const double *__restrict__ lam_v, int Bk, int Bv,
                                                    const int32_t *__restrict__ split,
                                                    int32_t *__restrict__ bits_k, int32_t *__restrict__ bits_v,
                                                    float *__restrict__ step_k, float *__restrict__ step_v,
                                                    StepTable steps)
{
    __shared__ double gain[D * AATC_MAXB];
    __shared__ double s_tab[AATC_MAXB + 1];
    __shared__ int nb[D];
    __shared__ unsigned long long mx;
    const int h = blockIdx.x, tensor = blockIdx.y, t = threadIdx.x;
    const double *lam = (tensor == 0 ? lam_k : lam_v) + h * D;
    const int B = split ? split[tensor] : (tensor == 0 ? Bk : Bv);
    if (t <= AATC_MAXB) s_tab[t] = steps.s[t];
    topB_alloc(lam, B, gain, nb, &mx);
    if (t < D) {
        int b = nb[t];
        (tensor == 0 ? bits_k : bits_v)[h * D + t] = b;
        float st = b > 0 ? (float)(s_tab[b] * sqrt(fmax(lam[t], 0.0))) : 0.0f;
        (tensor == 0 ? step_k : step_v)[h * D + t] = st;
    }
}

// Attention-aware token weights of each KV head ("Theorem: Additive Error
// Decomposition": value noise is weighted by A_i^2, key noise by
// A_i^2 |v_i - o|^2 and the query metric, which the key transform already
// holds):
//   alpha_V = mean_q sum_i A_qi^2,   alpha_K = mean_q (1/d) sum_i A_qi^2 |v_i - o_q|^2
// over the G N calibration queries of the head's group, each attending all N
// calibration keys of the head with the 1/sqrt(d) scale, no mask.  With
// e_i = 2^(s_i - m) (online maximum m), l = sum e, L2 = sum e^2,
// a = sum e v, a2 = sum e^2 v, n2 = sum e^2 |v|^2 (values centred by their
// calibration mean, which leaves v_i - o unchanged):
//   sum_i A_i^2 = L2 / l^2,
//   sum_i A_i^2 |v_i - o|^2 = (n2 - 2 (a . a2) / l + |a|^2 L2 / l^2) / l^2.
// One CTA per (64 queries, KV head); fp32 inside a query, fp64 across queries.
// Thread (tq, tk) scores queries 4tq.. against keys 4tk.. of a 64-key tile and
// then accumulates a and a2 of queries 4tq.. over channels 8tk.. .
constexpr int AQ = 64, AKT = 64, ATH = 256;
constexpr int QP = AQ + 4, KP = AKT + 4;   // padded rows of the transposed tiles (fewer bank conflicts)
constexpr size_t ALPHA_SMEM = (size_t)(D * QP + D * KP + AKT * D + AKT * AQ + AKT) * sizeof(float);

template <typename T>
__device__ __forceinline__ float ld_f32(const T *p) { return (float)to_f64(*p); }

template <typename T>
__global__ void __launch_bounds__(ATH) k_alpha(const T *__restrict__ k_cal, const T *__restrict__ v_cal,
                                               const T *__restrict__ q_cal, const double *__restrict__ mu_v, int N,
                                               int G, double *__restrict__ part)
{
    extern __shared__ __align__(16) float asm_[];
    float *Qt = asm_;                 // [D][QP]   queries, transposed
    float *Kt = Qt + D * QP;          // [D][KP]   keys, transposed
    float *Vs = Kt + D * KP;          // [AKT][D]  values minus their mean
    float *Pt = Vs + AKT * D;         // [AKT][AQ] e of (key, query)
    float *vn = Pt + AKT * AQ;        // [AKT]     |v|^2
    __shared__ double red[2][ATH / 32];
    const int h = blockIdx.y, qb = blockIdx.x, tid = threadIdx.x;
    const int tq = tid >> 4, tk = tid & 15;
    const long nq = (long)G * N;
    const float sc = 1.4426950408889634f / sqrtf((float)D);   // log2(e) / sqrt(d)
    // queries of this block: query n of the group is row n % N of query head h G + n / N
    for (int e = tid; e < AQ * D; e += ATH) {
        const int qi = e / D, kd = e % D;
        const long n = (long)qb * AQ + qi;
        float x = 0.f;
        if (n < nq) x = ld_f32(q_cal + ((size_t)(h * G + n / N) * N + n % N) * D + kd);
        Qt[kd * QP + qi] = x;
    }
    float m[4], l[4], L2[4], n2[4], a[4][8], a2[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        m[r] = -INFINITY;
        l[r] = L2[r] = n2[r] = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) a[r][c8] = a2[r][c8] = 0.f;
    }
    const T *Kh = k_cal + (size_t)h * N * D;
    const T *Vh = v_cal + (size_t)h * N * D;
    for (int k0 = 0; k0 < N; k0 += AKT) {
        __syncthreads();   // the previous tile is used up
        for (int e = tid; e < AKT * D; e += ATH) {
            const int ki = e / D, kd = e % D;
            const bool in = k0 + ki < N;
            Kt[kd * KP + ki] = in ? ld_f32(Kh + (size_t)(k0 + ki) * D + kd) : 0.f;
            Vs[ki * D + kd] = in ? (float)(to_f64(Vh[(size_t)(k0 + ki) * D + kd]) - mu_v[h * D + kd]) : 0.f;
        }
        __syncthreads();
        if (tid < AKT) {
            float s2 = 0.f;
            for (int kd = 0; kd < D; ++kd) s2 = fmaf(Vs[tid * D + kd], Vs[tid * D + kd], s2);
            vn[tid] = s2;
        }
        // scores of queries 4tq.. x keys 4tk.., log2 domain
        float sv[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) sv[r][c4] = 0.f;
#pragma unroll 4
        for (int kd = 0; kd < D; ++kd) {
            const float4 q4 = *reinterpret_cast<const float4 *>(&Qt[kd * QP + 4 * tq]);
            const float4 k4 = *reinterpret_cast<const float4 *>(&Kt[kd * KP + 4 * tk]);
            const float qq[4] = {q4.x, q4.y, q4.z, q4.w}, kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) sv[r][c4] = fmaf(qq[r], kk[c4], sv[r][c4]);
        }
        __syncthreads();   // vn is ready
        float f[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float tmax = -INFINITY;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                sv[r][c4] = k0 + 4 * tk + c4 < N ? sv[r][c4] * sc : -INFINITY;
                tmax = fmaxf(tmax, sv[r][c4]);
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            const float mn = fmaxf(m[r], tmax);
            f[r] = m[r] == -INFINITY ? 0.f : exp2f(m[r] - mn);
            m[r] = mn;
            float ls = 0.f, l2s = 0.f, n2s = 0.f;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const float e = exp2f(sv[r][c4] - mn);
                sv[r][c4] = e;
                ls += e;
                l2s = fmaf(e, e, l2s);
                n2s = fmaf(e * e, vn[4 * tk + c4], n2s);
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                ls += __shfl_xor_sync(0xffffffffu, ls, o);
                l2s += __shfl_xor_sync(0xffffffffu, l2s, o);
                n2s += __shfl_xor_sync(0xffffffffu, n2s, o);
            }
            l[r] = fmaf(l[r], f[r], ls);
            L2[r] = fmaf(L2[r], f[r] * f[r], l2s);
            n2[r] = fmaf(n2[r], f[r] * f[r], n2s);
        }
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
            *reinterpret_cast<float4 *>(&Pt[(4 * tk + c4) * AQ + 4 * tq]) =
                make_float4(sv[0][c4], sv[1][c4], sv[2][c4], sv[3][c4]);
        __syncthreads();
        // a, a2 of queries 4tq.. over channels 8tk..
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                a[r][c8] *= f[r];
                a2[r][c8] *= f[r] * f[r];
            }
        const int kn = min(AKT, N - k0);
        for (int ki = 0; ki < kn; ++ki) {
            const float4 p4 = *reinterpret_cast<const float4 *>(&Pt[ki * AQ + 4 * tq]);
            const float4 va = *reinterpret_cast<const float4 *>(&Vs[ki * D + 8 * tk]);
            const float4 vb = *reinterpret_cast<const float4 *>(&Vs[ki * D + 8 * tk + 4]);
            const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
            const float vv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float e2 = pp[r] * pp[r];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    a[r][c8] = fmaf(pp[r], vv[c8], a[r][c8]);
                    a2[r][c8] = fmaf(e2, vv[c8], a2[r][c8]);
                }
            }
        }
    }
    // per query: a . a2 and |a|^2 over the channels (16 threads per query group)
    double av = 0.0, ak = 0.0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        float d1 = 0.f, d2 = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            d1 = fmaf(a[r][c8], a2[r][c8], d1);
            d2 = fmaf(a[r][c8], a[r][c8], d2);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            d1 += __shfl_xor_sync(0xffffffffu, d1, o);
            d2 += __shfl_xor_sync(0xffffffffu, d2, o);
        }
        const long n = (long)qb * AQ + 4 * tq + r;
        if (tk == 0 && n < nq && l[r] > 0.f) {
            const double ld = l[r], il2 = 1.0 / (ld * ld);
            av += (double)L2[r] * il2;
            ak += ((double)n2[r] - 2.0 * (double)d1 / ld + (double)d2 * (double)L2[r] * il2) * il2 / D;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        av += __shfl_xor_sync(0xffffffffu, av, o);
        ak += __shfl_xor_sync(0xffffffffu, ak, o);
    }
    if ((tid & 31) == 0) {
        red[0][tid >> 5] = ak;
        red[1][tid >> 5] = av;
    }
    __syncthreads();
    if (tid < 2) {
        double sum = 0.0;
        for (int w = 0; w < ATH / 32; ++w) sum += red[tid][w];
        part[((size_t)h * gridDim.x + qb) * 2 + tid] = sum;
    }
}

// alpha[h][t] = sum over the query blocks / (G N).
__global__ void k_alpha_reduce(const double *__restrict__ part, int nqb, long nq, double *__restrict__ alpha)
{
    const int h = blockIdx.x, t = threadIdx.x;
    if (t >= 2) return;
    double s = 0.0;
    for (int b = 0; b < nqb; ++b) s += part[((size_t)h * nqb + b) * 2 + t];
    alpha[h * 2 + t] = s / (double)nq;
}

// Joint K/V budget split ("Theorem: Additive Error Decomposition" weights,
// "Optimal Bit Allocation via Reverse Water-Filling" over both tensors): for
// every word-aligned split B_K + B_V = Bpair (each 32..8 D) the exact top-B
// allocation of each head and tensor, and its distortion sum_j lam_j 4^{-b_j}.
// One block per (split, head, tensor).
__global__ void __launch_bounds__(1024) k_split_cost(const double *__restrict__ lam_k,
                                                     const double *__restrict__ lam_v, int Bk0, int Bpair,
                                                     double *__restrict__ cost)
{
    __shared__ double gain[D * AATC_MAXB];
    __shared__ int nb[D];
    __shared__ unsigned long long mx;
    __shared__ double red[32];
    const int c = blockIdx.x, h = blockIdx.y, tensor = blockIdx.z, t = threadIdx.x;
    const int H = gridDim.y;
    const int Bk = Bk0 + 32 * c, B = tensor == 0 ? Bk : Bpair - Bk;
    const double *lam = (tensor == 0 ? lam_k : lam_v) + h * D;
    topB_alloc(lam, B, gain, nb, &mx);
    double v = t < D ? ldexp(fmax(lam[t], 0.0), -2 * nb[t]) : 0.0;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((t & 31) == 0) red[t >> 5] = v;
    __syncthreads();
    if (t < 32) {
        v = red[t];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (t == 0) cost[((size_t)c * H + h) * 2 + tensor] = v;
    }
}

// The split of least sum_h alpha_Kh cost_K + alpha_Vh cost_V over the heads
// (ties to the split nearest Bpair / 2, then the smaller B_K) -> split[0] =
// B_K, split[1] = B_V.  One thread.
__global__ void k_split_pick(const double *__restrict__ cost, const double *__restrict__ alpha, int n_cand, int H,
                             int Bk0, int Bpair, int32_t *__restrict__ split)
{
    int best = -1;
    double best_c = 0.0;
    for (int c = 0; c < n_cand; ++c) {
        double tot = 0.0;
        for (int h = 0; h < H; ++h)
            tot += alpha[h * 2 + 0] * cost[((size_t)c * H + h) * 2 + 0] +
                   alpha[h * 2 + 1] * cost[((size_t)c * H + h) * 2 + 1];
        const int Bk = Bk0 + 32 * c;
        const bool better = best < 0 || tot < best_c ||
                            (tot == best_c && abs(2 * Bk - Bpair) < abs(2 * (Bk0 + 32 * best) - Bpair));
        if (better) {
            best = c;
            best_c = tot;
        }
    }
    split[0] = Bk0 + 32 * best;
    split[1] = Bpair - split[0];
}

// ---------------------------------------------------------------------------
// Derived fp32 operands and codec tables
// ---------------------------------------------------------------------------

// One block of 128 threads per (head, tensor): record layout offsets (all
// 8-bit fields, then 4-, 2-, 1-bit fields, channels ascending), 1/Delta,
// midpoints, and the bias b = T mu.
__global__ void k_tables(const int32_t *__restrict__ bits_k, const int32_t *__restrict__ bits_v,
                         const float *__restrict__ step_k, const float *__restrict__ step_v,
                         const double *__restrict__ T_k, const double *__restrict__ T_v,
                         const double *__restrict__ mu_k, const double *__restrict__ mu_v,
                         CodecTables *__restrict__ tab, float *__restrict__ bk32, float *__restrict__ bv32)
{
    const int h = blockIdx.x, tensor = blockIdx.y, j = threadIdx.x;
    const int32_t *bits = (tensor == 0 ? bits_k : bits_v) + h * D;
    const float *step = (tensor == 0 ? step_k : step_v) + h * D;
    CodecTables &T = tab[h * 2 + tensor];
    const int b = bits[j];
    const float st = step[j];
    T.bits[j] = (uint8_t)b;
    T.step[j] = st;
    T.inv_step[j] = b > 0 ? __frcp_rn(st) : 0.0f;
    T.mid[j] = b > 0 ? 0.5f * (float)((1 << b) - 1) : 0.0f;
    T.top[j] = (float)((1 << b) - 1);
    const double *Tm = (tensor == 0 ? T_k : T_v) + (size_t)h * D * D;
    const double *mu = (tensor == 0 ? mu_k : mu_v) + h * D;
    double acc = 0.0;
    for (int k = 0; k < D; ++k) acc += Tm[j * D + k] * mu[k];
    (tensor == 0 ? bk32 : bv32)[h * D + j] = (float)acc;
}

// y[h][c][r] = x[h][r][c] for H square [D][D] blocks (fp64 -> fp32, transposed)
__global__ void k_to_f32_t(const double *__restrict__ x, float *__restrict__ y)
{
    const int h = blockIdx.y, r = blockIdx.x, c = threadIdx.x;
    y[((size_t)h * D + c) * D + r] = (float)x[((size_t)h * D + r) * D + c];
}

// y[h][t][c][r] = T_t[h][r][c] in fp32: each head's two transforms, transposed, side by side
__global__ void k_to_f32_t2(const double *__restrict__ Tk, const double *__restrict__ Tv, float *__restrict__ y)
{
    const int h = blockIdx.y, t = blockIdx.z, r = blockIdx.x, c = threadIdx.x;
    const double *x = t ? Tv : Tk;
    y[(((size_t)h * 2 + t) * D + c) * D + r] = (float)x[((size_t)h * D + r) * D + c];
}

__global__ void k_to_f32(const double *__restrict__ x, float *__restrict__ y, size_t n)
{
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = (float)x[i];
}

template <typename T>
aatc_status launch_stats(const T *k, const T *v, const T *q, aatc_calib *h, int N, double *Sk,
                         double *Sv, double *Sq, double *partial, cudaStream_t s)
{
    const int H = h->Hkv, G = h->G;
    k_mean<T><<<H, D, 0, s>>>(k, N, h->mu_k, h->status);
    k_mean<T><<<H, D, 0, s>>>(v, N, h->mu_v, h->status);
    {   // q enters only through its second moment; check it for NaN/Inf
        const size_t nq = (size_t)h->Hq * N * D;
        const size_t blocks = (nq + 255) / 256 < 4096 ? (nq + 255) / 256 : 4096;
        k_check_finite<T><<<(unsigned)blocks, 256, 0, s>>>(q, nq, h->status);
    }
    const int nck = (N + MOMENT_CHUNK - 1) / MOMENT_CHUNK;
    const long nq = (long)G * N;
    const int nckq = (int)((nq + MOMENT_CHUNK - 1) / MOMENT_CHUNK);
    if (sizeof(T) == 2) {   // bf16: exact digit-split contraction on the tensor cores
        const __nv_bfloat16 *kb = reinterpret_cast<const __nv_bfloat16 *>(k);
        const __nv_bfloat16 *vb = reinterpret_cast<const __nv_bfloat16 *>(v);
        const __nv_bfloat16 *qb = reinterpret_cast<const __nv_bfloat16 *>(q);
        aatc_status st = cov_tc_run(kb, H, N, h->mu_k, Sk, N, partial, h->status, s);
        if (st == AATC_OK) st = cov_tc_run(vb, H, N, h->mu_v, Sv, N, partial, h->status, s);
        if (st == AATC_OK) st = cov_tc_run(qb, H, nq, nullptr, Sq, nq, partial, h->status, s);
        return st;
    }
    k_moment_partial<T><<<dim3(nck, H), 256, 0, s>>>(k, N, h->mu_k, partial);
    k_moment_reduce<<<dim3(D * D / 256, H), 256, 0, s>>>(partial, nck, N, Sk);
    k_moment_partial<T><<<dim3(nck, H), 256, 0, s>>>(v, N, h->mu_v, partial);
    k_moment_reduce<<<dim3(D * D / 256, H), 256, 0, s>>>(partial, nck, N, Sv);
    k_moment_partial<T><<<dim3(nckq, H), 256, 0, s>>>(q, nq, nullptr, partial);
    k_moment_reduce<<<dim3(D * D / 256, H), 256, 0, s>>>(partial, nckq, nq, Sq);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

}  // namespace

size_t calib_work_bytes(int Hkv, int Hq, int N)
{
    const int G = Hq / Hkv;
    const size_t mat = (size_t)D * D * sizeof(double);
    const size_t nck = (size_t)(N + MOMENT_CHUNK - 1) / MOMENT_CHUNK;
    const size_t nckq = ((size_t)G * N + MOMENT_CHUNK - 1) / MOMENT_CHUNK;
    size_t partial = (size_t)Hkv * (nck > nckq ? nck : nckq) * mat;
    const size_t tc = cov_tc_scratch(Hkv, (long)G * N);   // the largest of the three (rows G N >= N)
    if (tc > partial) partial = tc;
    partial = (partial + 255) & ~(size_t)255;
    return partial + (size_t)Hkv * 13 * mat;   // Sk Sv Sq Uq Sh Si Mk, Jacobi scratch 3 x 2H
}

// Eigendecomposition of m symmetric matrices A[m] (fp64), the first M0 into
// (evals0, evecs0), the rest into (evals1, evecs1): fp32 sweeps give the
// rotations Q; two Newton-Schulz steps make Q orthogonal in fp64
// (Q <- Q (3 I - Q^T Q) / 2); the fp64 sweeps run on Q^T A Q, accumulating from Q.
static aatc_status jacobi_mixed(const double *A, int m, int M0, double *evals0, double *evecs0, double *evals1,
                         double *evecs1, double *Q, double *X, double *Y, int max_sweeps, uint32_t *status,
                         cudaStream_t s)
{
    constexpr size_t M = (size_t)D * D;
    AATC_CUDA(cudaFuncSetAttribute(k_jacobi<float, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)jac_smem<float>()));
    AATC_CUDA(cudaFuncSetAttribute(k_jacobi<double, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)jac_smem<double>()));
    k_jacobi<float, true><<<m, JAC_THREADS, jac_smem<float>(), s>>>(A, nullptr, Q, nullptr, m, nullptr, nullptr,
                                                                    nullptr, nullptr, PRE_SWEEPS, status);
    const dim3 gg(D * D / 256, m);
    const size_t n = (size_t)m * M;
    for (int it = 0; it < 2; ++it) {
        k_gemm64<<<gg, 256, 0, s>>>(Q, 1, nullptr, DIAG_NONE, Q, 0, X);   // X = Q^T Q
        k_gemm64<<<gg, 256, 0, s>>>(Q, 0, nullptr, DIAG_NONE, X, 0, Y);   // Y = Q X
        k_ns_step<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(Q, Y, n);
    }
    k_gemm64<<<gg, 256, 0, s>>>(Q, 1, nullptr, DIAG_NONE, A, 0, X);       // X = Q^T A
    k_gemm64<<<gg, 256, 0, s>>>(X, 0, nullptr, DIAG_NONE, Q, 0, Y);       // Y = Q^T A Q
    k_jacobi<double, false><<<m, JAC_THREADS, jac_smem<double>(), s>>>(Y, evals0, evecs0, Q, M0, Y + M0 * M,
                                                                       evals1, evecs1, Q + M0 * M, max_sweeps,
                                                                       status);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

aatc_status calib_run(aatc_calib *h, const void *k_cal, const void *v_cal, const void *q_cal,
                      int N, int max_sweeps, void *work, cudaStream_t s)
{
    const int H = h->Hkv;
    const size_t M = (size_t)D * D;
    double *base = (double *)work;
    const int G = h->G;
    const size_t nck = (size_t)(N + MOMENT_CHUNK - 1) / MOMENT_CHUNK;
    const size_t nckq = ((size_t)G * N + MOMENT_CHUNK - 1) / MOMENT_CHUNK;
    double *partial = base;
    size_t pbytes = (size_t)H * (nck > nckq ? nck : nckq) * M * sizeof(double);
    const size_t tc = cov_tc_scratch(H, (long)G * N);
    if (tc > pbytes) pbytes = tc;
    pbytes = (pbytes + 255) & ~(size_t)255;
    double *Sk = (double *)((char *)base + pbytes);
    double *Sv = Sk + H * M, *Sq = Sv + H * M, *Uq = Sq + H * M, *Sh = Uq + H * M,
           *Si = Sh + H * M, *Mk = Si + H * M;
    double *Qs = Mk + H * M, *Xs = Qs + 2 * H * M, *Ys = Xs + 2 * H * M;   // Jacobi scratch, 2H each
    aatc_status st;
    if (h->dtype == AATC_BF16)
        st = launch_stats((const __nv_bfloat16 *)k_cal, (const __nv_bfloat16 *)v_cal,
                          (const __nv_bfloat16 *)q_cal, h, N, Sk, Sv, Sq, partial, s);
    else
        st = launch_stats((const float *)k_cal, (const float *)v_cal, (const float *)q_cal, h, N,
                          Sk, Sv, Sq, partial, s);
    if (st != AATC_OK) return st;

    // query metric: Sq = Uq Lq Uq^T ; Sh = Sq^{1/2}, Si = Sq^{-1/2}; with it the
    // value KLT Sv = Uv Lv Uv^T (independent of the key path).  Sv and Sq are
    // adjacent: one batch of 2H matrices.
    st = jacobi_mixed(Sv, 2 * H, H, h->lam_v, h->U_v, h->lam_q, Uq, Qs, Xs, Ys, max_sweeps, h->status, s);
    if (st != AATC_OK) return st;
    const dim3 gg(D * D / 256, H);
    k_gemm64<<<gg, 256, 0, s>>>(Uq, 0, h->lam_q, DIAG_SQRT, Uq, 1, Sh);
    k_gemm64<<<gg, 256, 0, s>>>(Uq, 0, h->lam_q, DIAG_INVSQRT, Uq, 1, Si);
    // whitened key covariance Mk = Sh Sk Sh (Jacobi reads its symmetric part)
    k_gemm64<<<gg, 256, 0, s>>>(Sh, 0, nullptr, DIAG_NONE, Sk, 0, Uq);       // Uq reused as tmp
    k_gemm64<<<gg, 256, 0, s>>>(Uq, 0, nullptr, DIAG_NONE, Sh, 0, Mk);
    // key KLT: Mk = Uk Lk Uk^T (Uk kept in Uq)
    st = jacobi_mixed(Mk, H, H, h->lam_k, Uq, nullptr, nullptr, Qs, Xs, Ys, max_sweeps, h->status, s);
    if (st != AATC_OK) return st;
    // Tk = Uk^T Sh, Ak = Uk^T Si, Tk^{-1} = Si Uk, Tv = Uv^T
    k_gemm64<<<gg, 256, 0, s>>>(Uq, 1, nullptr, DIAG_NONE, Sh, 0, h->T_k);
    k_gemm64<<<gg, 256, 0, s>>>(Uq, 1, nullptr, DIAG_NONE, Si, 0, h->A_k);
    k_gemm64<<<gg, 256, 0, s>>>(Si, 0, nullptr, DIAG_NONE, Uq, 0, h->T_k_inv);
    k_transpose64<<<gg, 256, 0, s>>>(h->U_v, h->T_v);
    AATC_CUDA(cudaGetLastError());
    const int32_t *split = nullptr;
    if (h->joint) {
        // joint allocation: the token weights of the calibration attention, then
        // the word-aligned split of the pair budget (each tensor 32 .. 8 D bits)
        // of least weighted distortion over the heads; the moment partials'
        // scratch is free by now
        const int nqb = (G * N + AQ - 1) / AQ;
        double *apart = partial;
        double *cost = apart + (size_t)H * nqb * 2;
        const int Bk0 = h->Bpair - AATC_MAXB * D > 32 ? h->Bpair - AATC_MAXB * D : 32;
        const int Bk1 = h->Bpair - 32 < AATC_MAXB * D ? h->Bpair - 32 : AATC_MAXB * D;
        if (Bk1 < Bk0) return aatc_fail(AATC_ERR_UNSUPPORTED, "pair budget of %d bits cannot be split", h->Bpair);
        const int n_cand = (Bk1 - Bk0) / 32 + 1;
        if (h->dtype == AATC_BF16) {
            st = kernel_smem_limit((const void *)k_alpha<__nv_bfloat16>, ALPHA_SMEM);
            if (st != AATC_OK) return st;
            k_alpha<__nv_bfloat16><<<dim3(nqb, H), ATH, ALPHA_SMEM, s>>>(
                (const __nv_bfloat16 *)k_cal, (const __nv_bfloat16 *)v_cal, (const __nv_bfloat16 *)q_cal, h->mu_v, N,
                G, apart);
        } else {
            st = kernel_smem_limit((const void *)k_alpha<float>, ALPHA_SMEM);
            if (st != AATC_OK) return st;
            k_alpha<float><<<dim3(nqb, H), ATH, ALPHA_SMEM, s>>>((const float *)k_cal, (const float *)v_cal,
                                                               (const float *)q_cal, h->mu_v, N, G, apart);
        }
        k_alpha_reduce<<<H, 32, 0, s>>>(apart, nqb, (long)G * N, h->alpha);
        k_split_cost<<<dim3(n_cand, H, 2), 1024, 0, s>>>(h->lam_k, h->lam_v, Bk0, h->Bpair, cost);
        k_split_pick<<<1, 1, 0, s>>>(cost, h->alpha, n_cand, H, Bk0, h->Bpair, h->split);
        AATC_CUDA(cudaGetLastError());
        split = h->split;
    }
    k_waterfill<<<dim3(H, 2), 1024, 0, s>>>(h->lam_k, h->lam_v, h->Bk, h->Bv, split, h->bits_k, h->bits_v,
                                            h->step_k, h->step_v, step_table());
    AATC_CUDA(cudaGetLastError());
    return calib_derive(h, s);
}

aatc_status calib_derive(aatc_calib *h, cudaStream_t s)
{
    const int H = h->Hkv;
    const size_t n = (size_t)H * D * D;
    const int blocks = (int)((n + 255) / 256);
    k_to_f32<<<blocks, 256, 0, s>>>(h->T_k, h->Tk32, n);
    k_to_f32<<<blocks, 256, 0, s>>>(h->T_v, h->Tv32, n);
    k_to_f32_t<<<dim3(D, H), D, 0, s>>>(h->A_k, h->AkT32);
    k_to_f32_t<<<dim3(D, H), D, 0, s>>>(h->U_v, h->UvT32);
    k_to_f32_t2<<<dim3(D, H, 2), D, 0, s>>>(h->T_k, h->T_v, h->TkvT32);
    k_to_f32<<<(H * D + 255) / 256, 256, 0, s>>>(h->mu_v, h->muv32, (size_t)H * D);
    k_tables<<<dim3(H, 2), D, 0, s>>>(h->bits_k, h->bits_v, h->step_k, h->step_v, h->T_k, h->T_v,
                                      h->mu_k, h->mu_v, h->tab, h->bk32, h->bv32);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

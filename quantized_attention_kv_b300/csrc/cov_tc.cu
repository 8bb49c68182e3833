// cov_tc.cu -- calibration second moments on the tensor cores.
//
// Sigma = (1/n) sum_t (x_t - c)(x_t - c)^T for the key/value covariances
// (c = mean) and the pooled query second moment (c = 0) ("Attention-Aware
// Transform Coding Guide: KV Compression", section "Decorrelation via the
// Karhunen-Loeve Transform (KLT)"; the query weighting of section "Theorem:
// Additive Error Decomposition").
//
// The contraction is made exact so that the fp64 eigensolver downstream sees
// the covariance of the data to within one rounding of the input:
//   1. d = x - c is rounded once to a 28-bit fixed-point integer
//      n = rint(d 2^s_j), with one power-of-two scale 2^s_j per (matrix,
//      head, channel j) chosen so that |n| < 2^27;
//   2. n is split into four balanced 7-bit digits, n = sum_p D_p 2^(7p) with
//      |D_p| <= 64, each an integer that bf16 holds exactly;
//   3. for each digit pair (p, q), sum_t D_p(t) D_q(t)^T runs on tcgen05.mma
//      (bf16 in, fp32 accumulation in tensor memory) over at most 1024
//      tokens: every partial sum is an integer below 2^24, so fp32 carries it
//      without rounding, whatever order the hardware adds in;
//   4. the chunks and digit pairs are summed in fp64 with their 2^(7(p+q))
//      weights and the 2^(-s_i - s_j) scales.
// Pairs with the same p + q share one accumulator (at most four pairs, still
// below 2^24): p + q = 0..3 in a first pass over the chunk, 4..6 in a second.
#include <cuda_bf16.h>

#include "internal.h"
#include "tc_util.h"

namespace {

using namespace tc;

constexpr int D = AATC_D;
constexpr int CT_TOK = 64;                   // tokens per tile (one 128-byte swizzled K row)
constexpr int CT_TILES = 16;                 // tiles per CTA: 1024 tokens keep the sums exact
constexpr int NDIG = 4;                      // digits of 7 bits
constexpr int NK = 2 * NDIG - 1;             // distinct p + q
constexpr uint32_t PLANE_BYTES = D * CT_TOK * 2;                 // 16 KB
constexpr uint32_t STAGE_BYTES = NDIG * PLANE_BYTES;             // 64 KB
constexpr size_t CT_SMEM = 1024 + 2 * (size_t)STAGE_BYTES;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// amax_bits[h][j] = bits of max |x_j - c_j| over head h's rows (non-negative
// floats order like their bit patterns).  X: [H][T][D].
template <typename T>
__global__ void k_cov_absmax(const T *__restrict__ X, long rows, const double *__restrict__ center,
                             unsigned int *__restrict__ amax_bits)
{
    __shared__ unsigned int bm[D];
    const int h = blockIdx.y, j = threadIdx.x & (D - 1);
    if (threadIdx.x < D) bm[threadIdx.x] = 0u;
    __syncthreads();
    const double cj = center ? center[h * D + j] : 0.0;
    const T *x = X + (size_t)h * rows * D;
    float m = 0.f;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < (size_t)rows * D;
         e += (size_t)gridDim.x * blockDim.x)
        m = fmaxf(m, (float)fabs((double)to_f32(x[e]) - cj));   // blockDim and the stride are multiples of D
    atomicMax(&bm[j], __float_as_uint(m));
    __syncthreads();
    if (threadIdx.x < D) atomicMax(&amax_bits[h * D + threadIdx.x], bm[threadIdx.x]);
}

// Scale exponent s with max|x - c| * 2^s < 2^27 (0 when the data are all equal to c).
__device__ __forceinline__ int cov_scale_exp(unsigned int amax_bits)
{
    const float a = __uint_as_float(amax_bits);
    if (!(a > 0.f)) return 0;
    int e;
    frexpf(a * 1.0000001f, &e);   // a < 2^e (the factor covers the float rounding of |x - c|)
    return 27 - e;
}

// Digits of rint((x_j - c_j) 2^s_j), transposed: dig[h][p][channel][token]
// (bf16, tokens padded to Tpad with zeros).  One block per 64 tokens of one head.
template <typename T>
__global__ void __launch_bounds__(256) k_cov_digits(const T *__restrict__ X, long rows, long Tpad,
                                                    const double *__restrict__ center,
                                                    const unsigned int *__restrict__ amax_bits,
                                                    int *__restrict__ sexp, __nv_bfloat16 *__restrict__ dig)
{
    __shared__ int ns[CT_TOK][D + 1];
    const int h = blockIdx.y, tid = threadIdx.x;
    const long t0 = (long)blockIdx.x * CT_TOK;
    const int j = tid & (D - 1);   // every element this thread rounds is channel j (256 = 2 D)
    const int s = cov_scale_exp(amax_bits[h * D + j]);
    if (blockIdx.x == 0 && tid < D) sexp[h * D + j] = s;
    const double scale = ldexp(1.0, s), cj = center ? center[h * D + j] : 0.0;
    const T *x = X + (size_t)h * rows * D;
    for (int e = tid; e < CT_TOK * D; e += 256) {
        const int i = e >> 7;
        const long t = t0 + i;
        int n = 0;
        if (t < rows) n = (int)rint(((double)to_f32(x[(size_t)t * D + j]) - cj) * scale);
        ns[i][j] = n;
    }
    __syncthreads();
    // thread (channel j, token pair tp): balanced digits of tokens 2tp, 2tp+1
    for (int e = tid; e < D * (CT_TOK / 2); e += 256) {
        const int jj = e >> 5, tp = e & 31;
        int a = ns[2 * tp][jj], b = ns[2 * tp + 1][jj];
#pragma unroll
        for (int p = 0; p < NDIG; ++p) {
            int da = a, db = b;
            if (p < NDIG - 1) {
                da = ((a + 64) & 127) - 64;
                db = ((b + 64) & 127) - 64;
                a = (a - da) >> 7;
                b = (b - db) >> 7;
            }
            __nv_bfloat162 v;
            v.x = __int2bfloat16_rn(da);
            v.y = __int2bfloat16_rn(db);
            *reinterpret_cast<__nv_bfloat162 *>(dig + (((size_t)h * NDIG + p) * D + jj) * Tpad + t0 + 2 * tp) = v;
        }
    }
}

// Digit-pair sums over one chunk of up to CT_TILES tiles of one head:
// part[h][chunk][k][i][j] = sum over p + q = k, t in chunk of D_p(t)_i D_q(t)_j
// (exact integers in fp32).  128 threads: thread 0 issues the loads and the
// MMAs; all four warps read tensor memory (thread = row i).
__global__ void __launch_bounds__(128, 1) k_cov_tc(const __grid_constant__ CUtensorMap map, int ntiles,
                                                   int nchunk, float *__restrict__ part, uint32_t *status)
{
    extern __shared__ unsigned char sm_raw[];
    // 1024-byte aligned in the shared window; derived from sm_raw by pointer arithmetic so that
    // every access through it compiles to a shared-memory instruction
    unsigned char *sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) uint64_t full[2], empty[2], done;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x, h = blockIdx.y;
    const int kt0 = chunk * CT_TILES, n = min(CT_TILES, ntiles - kt0);
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_base;
    bool ok = true;
    int g0 = 0;   // tiles consumed so far (both passes): tile g uses stage g & 1, phase (g >> 1) & 1
    for (int pass = 0; pass < 2; ++pass) {
        const int kbase = pass ? NDIG : 0, nk = pass ? NK - NDIG : NDIG;
        if (tid == 0) {
            auto issue = [&](int g, int j) {
                const int s = g & 1;
                mbar_expect(&full[s], STAGE_BYTES);
                for (int p = 0; p < NDIG; ++p)
                    tma2d(sm + s * STAGE_BYTES + p * PLANE_BYTES, &map, (kt0 + j) * CT_TOK, (h * NDIG + p) * D, &full[s]);
            };
            for (int j = 0; j < 2 && j < n && ok; ++j) issue(g0 + j, j);
            bool started[NDIG] = {false, false, false, false};
            for (int j = 0; j < n && ok; ++j) {
                const int g = g0 + j, s = g & 1;
                ok = mbar_wait1(&full[s], (uint32_t)((g >> 1) & 1));
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t base = smem_u32(sm + s * STAGE_BYTES);
                for (int p = 0; p < NDIG; ++p)
                    for (int q = 0; q < NDIG; ++q) {
                        const int k = p + q - kbase;
                        if (k < 0 || k >= nk) continue;
                        const uint32_t dcol = tmem + k * D;
#pragma unroll
                        for (int ks = 0; ks < CT_TOK / 16; ++ks) {
                            mma_bf16(dcol, desc_sw128(base + p * PLANE_BYTES + ks * 32),
                                     desc_sw128(base + q * PLANE_BYTES + ks * 32), started[k] ? 1u : 0u);
                            started[k] = true;
                        }
                    }
                mma_commit(&empty[s]);
                // refill the stage the previous tile used
                if (j >= 1 && j + 1 < n) {
                    const int gp = g - 1;
                    ok = mbar_wait1(&empty[gp & 1], (uint32_t)((gp >> 1) & 1));
                    if (ok) issue(gp + 2, j + 1);
                }
            }
            mma_commit(&done);
        }
        // all tiles of the pass are in the accumulators once `done` completes
        if (!mbar_wait1(&done, (uint32_t)(pass & 1))) ok = false;
        asm volatile("tcgen05.fence::after_thread_sync;");
        const int i = warp * 32 + lane;
        for (int k = 0; k < nk; ++k) {
            float *dst = part + ((((size_t)h * nchunk + chunk) * NK + kbase + k) * D + i) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + k * D + c0, r);
                tmem_wait_ld(r);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<float4 *>(dst + c0 + 4 * q4) =
                        ok ? make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                                         __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        asm volatile("tcgen05.fence::before_thread_sync;");
        __syncthreads();
        g0 += n;
    }
    if (!ok && tid == 0) atomicOr(status, AATC_DEV_TIMEOUT);
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
}

// S[h][i][j] = 2^(-s_i - s_j) / count * sum over chunks, k of 2^(7k) part[h][chunk][k][i][j]  (fp64)
__global__ void k_cov_combine(const float *__restrict__ part, int nchunk, const int *__restrict__ sexp,
                              long count, double *__restrict__ S)
{
    const int h = blockIdx.y, e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= D * D) return;
    double acc[NK] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};
    for (int c = 0; c < nchunk; ++c)
#pragma unroll
        for (int k = 0; k < NK; ++k) acc[k] += (double)part[(((size_t)h * nchunk + c) * NK + k) * D * D + e];
    double s = 0.0;
#pragma unroll
    for (int k = NK - 1; k >= 0; --k) s += ldexp(acc[k], 7 * k);
    S[(size_t)h * D * D + e] = ldexp(s, -sexp[h * D + (e >> 7)] - sexp[h * D + (e & (D - 1))]) / (double)count;
}

}  // namespace

size_t cov_tc_scratch(int H, long rows)
{
    const long Tpad = (rows + CT_TOK - 1) / CT_TOK * CT_TOK;
    const long ntiles = Tpad / CT_TOK;
    const long nchunk = (ntiles + CT_TILES - 1) / CT_TILES;
    const size_t dig = (size_t)H * NDIG * D * Tpad * 2;
    const size_t part = (size_t)H * nchunk * NK * D * D * 4;
    return ((dig + 1023) & ~(size_t)1023) + part + (size_t)H * D * 8 + 1024;
}

aatc_status cov_tc_run(const __nv_bfloat16 *X, int H, long rows, const double *center, double *S, long count,
                       void *scratch, uint32_t *status, cudaStream_t s)
{
    const long Tpad = (rows + CT_TOK - 1) / CT_TOK * CT_TOK;
    const int ntiles = (int)(Tpad / CT_TOK);
    const int nchunk = (ntiles + CT_TILES - 1) / CT_TILES;
    const size_t dig_bytes = (size_t)H * NDIG * D * Tpad * 2;
    __nv_bfloat16 *dig = (__nv_bfloat16 *)scratch;
    float *part = (float *)((char *)scratch + ((dig_bytes + 1023) & ~(size_t)1023));
    unsigned int *amax = (unsigned int *)((char *)part + (size_t)H * nchunk * NK * D * D * 4);   // [H][D]
    int *sexp = (int *)(amax + (size_t)H * D);                                                   // [H][D]
    alignas(64) unsigned char map[128];
    if (!tma_map_bf16(map, dig, (unsigned long long)Tpad, (unsigned long long)H * NDIG * D))
        return aatc_fail(AATC_ERR_CUDA, "cuTensorMapEncodeTiled failed for the covariance digits");
    AATC_CUDA(cudaMemsetAsync(amax, 0, (size_t)H * D * sizeof(unsigned int), s));
    k_cov_absmax<__nv_bfloat16><<<dim3(64, H), 256, 0, s>>>(X, rows, center, amax);
    k_cov_digits<__nv_bfloat16><<<dim3((unsigned)(Tpad / CT_TOK), H), 256, 0, s>>>(X, rows, Tpad, center, amax, sexp,
                                                                                  dig);
    AATC_CUDA(cudaFuncSetAttribute(k_cov_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CT_SMEM));
    CUtensorMap m;
    memcpy(&m, map, sizeof(m));
    k_cov_tc<<<dim3(nchunk, H), 128, CT_SMEM, s>>>(m, ntiles, nchunk, part, status);
    k_cov_combine<<<dim3(D * D / 256, H), 256, 0, s>>>(part, nchunk, sexp, count, S);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

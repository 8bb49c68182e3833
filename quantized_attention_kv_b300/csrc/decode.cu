// decode.cu -- decode attention over the packed cache.
//
// o = softmax(q K^T / sqrt(d)) V ("Attention-Aware Transform Coding Guide:
// KV Compression", section "Formal Attention Distortion Model"), computed
// without reconstructing K or V:
//   score_i = q . k_hat_i / sqrt(d) = q' . u_i + const,  q' = (Tk^{-T} q) o Delta_K / sqrt(d)
// (the key mean and the code midpoints add the same constant to every score
// and cancel in the softmax), values are accumulated as codes in the
// transform domain, and the inverse value transform is applied once per head:
//   o = Uv (Delta_V o (sum_i p_i u_i / sum_i p_i - mid)) + mu_v.
// Decoding is bandwidth-bound ("Spend Bits Where Queries Look", Abstract):
// the kernels stream each packed record once.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace {

constexpr int D = AATC_D;
constexpr int DEC_TILE = 128;   // tokens per tile, one thread per token
constexpr int DEC_TARGET_BLOCKS = 2 * 148;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

struct SplitPlan {
    int n_split;   // blocks per (batch row, KV head)
    int chunk;     // tokens per block (multiple of DEC_TILE)
};

SplitPlan plan_splits(int B, int Hkv, int L)
{
    SplitPlan p;
    int tiles = (L + DEC_TILE - 1) / DEC_TILE;
    if (tiles < 1) tiles = 1;
    int want = (DEC_TARGET_BLOCKS + B * Hkv - 1) / (B * Hkv);
    if (want < 1) want = 1;
    if (want > tiles) want = tiles;
    int tiles_per = (tiles + want - 1) / want;
    p.chunk = tiles_per * DEC_TILE;
    p.n_split = (tiles + tiles_per - 1) / tiles_per;
    return p;
}

// q'[b][hq][j] = (A_k q)_j * Delta_K,j / sqrt(D), 0 for pruned channels.
template <typename T>
__global__ void k_query_prep(const T *__restrict__ q, int Hq, int G, const float *__restrict__ Ak,
                             const CodecTables *__restrict__ tabs, float *__restrict__ qp)
{
    __shared__ float qs[D];
    const int b = blockIdx.x, hq = blockIdx.y, j = threadIdx.x;
    const int h = hq / G;
    qs[j] = to_f32(q[((size_t)b * Hq + hq) * D + j]);
    __syncthreads();
    const float *A = Ak + (size_t)h * D * D + (size_t)j * D;
    float acc = 0.f;
    for (int k = 0; k < D; ++k) acc = fmaf(A[k], qs[k], acc);
    const CodecTables &tb = tabs[h * 2 + 0];
    qp[((size_t)b * Hq + hq) * D + j] = tb.bits[j] ? acc * tb.step[j] * 0.08838834764831845f : 0.f;
}

__device__ __forceinline__ uint32_t unpack_code(const uint32_t *rec, const int16_t (*off)[4], int bj, int j)
{
    uint32_t u = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int o = off[j][s];
        if (o >= 0) {
            const int width = 1 << s;
            const uint32_t f = (rec[o >> 5] >> (o & 31)) & ((1u << width) - 1u);
            u |= f << (bj & (width - 1));
        }
    }
    return u;
}

// One block per (split, KV head, batch row): online softmax over the block's
// token range for the G query heads of the KV head.  Partials per query head:
// m (running max of scores), l (sum of exp), acc[j] = sum_i p_i u^V_ij.
__global__ void __launch_bounds__(DEC_TILE) k_decode_split_simple(
    const float *__restrict__ qp, const uint32_t *__restrict__ kp, const uint32_t *__restrict__ vp,
    int L_cap, const int32_t *__restrict__ seq_lens, int L, int Hkv, int G, int W, int chunk,
    int n_split, const CodecTables *__restrict__ tabs, float *__restrict__ part)
{
    __shared__ float q_s[AATC_MAX_G][D];
    __shared__ float p_s[DEC_TILE][AATC_MAX_G + 1];
    __shared__ uint8_t v_s[DEC_TILE][D + 4];
    __shared__ int16_t offk[D][4], offv[D][4];
    __shared__ uint8_t bk[D], bv[D];
    __shared__ float red[4][AATC_MAX_G];
    __shared__ float m_s[AATC_MAX_G], alpha_s[AATC_MAX_G];

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    const int len = seq_lens ? min(max(seq_lens[b], 0), L) : L;
    const int begin = split * chunk, end = min(begin + chunk, len);
    const int Hq = Hkv * G;
    for (int e = t; e < G * D; e += DEC_TILE) {
        int g = e / D, j = e % D;
        q_s[g][j] = qp[((size_t)b * Hq + h * G + g) * D + j];
    }
    {
        const CodecTables &tk = tabs[h * 2 + 0], &tv = tabs[h * 2 + 1];
        for (int s = 0; s < 4; ++s) { offk[t][s] = tk.off[t][s]; offv[t][s] = tv.off[t][s]; }
        bk[t] = tk.bits[t];
        bv[t] = tv.bits[t];
    }
    if (t < AATC_MAX_G) m_s[t] = -INFINITY;
    __syncthreads();

    float acc[AATC_MAX_G], lsum[AATC_MAX_G];
#pragma unroll
    for (int g = 0; g < AATC_MAX_G; ++g) { acc[g] = 0.f; lsum[g] = 0.f; }

    const size_t base = ((size_t)b * Hkv + h) * L_cap;
    for (int tok0 = begin; tok0 < end; tok0 += DEC_TILE) {
        const int tok = tok0 + t;
        const bool valid = tok < end;
        uint32_t rec[32];
        float sc[AATC_MAX_G];
#pragma unroll
        for (int g = 0; g < AATC_MAX_G; ++g) sc[g] = -INFINITY;
        if (valid) {
            const uint32_t *r = kp + (base + tok) * W;
            for (int w = 0; w < W; ++w) rec[w] = r[w];
#pragma unroll
            for (int g = 0; g < AATC_MAX_G; ++g) sc[g] = 0.f;
            for (int j = 0; j < D; ++j) {
                if (!bk[j]) continue;
                const float u = (float)unpack_code(rec, offk, bk[j], j);
#pragma unroll
                for (int g = 0; g < AATC_MAX_G; ++g)
                    if (g < G) sc[g] = fmaf(q_s[g][j], u, sc[g]);
            }
            const uint32_t *rv = vp + (base + tok) * W;
            for (int w = 0; w < W; ++w) rec[w] = rv[w];
            for (int j = 0; j < D; ++j) v_s[t][j] = bv[j] ? (uint8_t)unpack_code(rec, offv, bv[j], j) : 0;
        } else {
            for (int j = 0; j < D; ++j) v_s[t][j] = 0;
        }
        // tile max per query head
#pragma unroll
        for (int g = 0; g < AATC_MAX_G; ++g) {
            float mx = sc[g];
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) red[warp][g] = mx;
        }
        __syncthreads();
        if (t < G) {
            float mx = fmaxf(fmaxf(red[0][t], red[1][t]), fmaxf(red[2][t], red[3][t]));
            float mo = m_s[t], mn = fmaxf(mo, mx);
            alpha_s[t] = (mo == -INFINITY) ? 0.f : __expf(mo - mn);
            m_s[t] = mn;
        }
        __syncthreads();
#pragma unroll
        for (int g = 0; g < AATC_MAX_G; ++g)
            if (g < G) p_s[t][g] = valid ? __expf(sc[g] - m_s[g]) : 0.f;
        __syncthreads();
        // thread t now owns value channel j = t
#pragma unroll
        for (int g = 0; g < AATC_MAX_G; ++g)
            if (g < G) { acc[g] *= alpha_s[g]; lsum[g] *= alpha_s[g]; }
        for (int i = 0; i < DEC_TILE; ++i) {
            const float u = (float)v_s[i][t];
#pragma unroll
            for (int g = 0; g < AATC_MAX_G; ++g)
                if (g < G) { acc[g] = fmaf(p_s[i][g], u, acc[g]); lsum[g] += p_s[i][g]; }
        }
        __syncthreads();
    }
    // partial layout [B][Hq][n_split][2 + D]: m, l, acc[D]
#pragma unroll
    for (int g = 0; g < AATC_MAX_G; ++g) {
        if (g >= G) break;
        float *P = part + (((size_t)b * Hq + h * G + g) * n_split + split) * (2 + D);
        P[2 + t] = acc[g];
        if (t == 0) { P[0] = m_s[g]; P[1] = lsum[g]; }
    }
}

// One block per (batch row, query head): LSE-merge the splits, leave the
// transform domain, apply Uv and add mu_v.  A row with no tokens gets zeros.
__global__ void k_decode_combine(const float *__restrict__ part, int n_split, int Hq, int G,
                                 const CodecTables *__restrict__ tabs, const float *__restrict__ Uv,
                                 const float *__restrict__ muv, float *__restrict__ out)
{
    __shared__ float cbar[D];
    const int b = blockIdx.x, hq = blockIdx.y, j = threadIdx.x;
    const int h = hq / G;
    const float *P = part + ((size_t)b * Hq + hq) * n_split * (2 + D);
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, P[s * (2 + D)]);
    float l = 0.f, a = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < n_split; ++s) {
            const float ms = P[s * (2 + D)];
            if (ms == -INFINITY) continue;
            const float w = __expf(ms - M);
            l = fmaf(P[s * (2 + D) + 1], w, l);
            a = fmaf(P[s * (2 + D) + 2 + j], w, a);
        }
    }
    const CodecTables &tv = tabs[h * 2 + 1];
    cbar[j] = (l > 0.f && tv.bits[j]) ? tv.step[j] * (a / l - tv.mid[j]) : 0.f;
    __syncthreads();
    float o = 0.f;
    if (l > 0.f) {
        const float *U = Uv + (size_t)h * D * D + (size_t)j * D;
        for (int k = 0; k < D; ++k) o = fmaf(U[k], cbar[k], o);
        o += muv[h * D + j];
    }
    out[((size_t)b * Hq + hq) * D + j] = o;
}

}  // namespace

size_t decode_ws_bytes(const aatc_calib *h, int B, int L)
{
    SplitPlan p = plan_splits(B, h->Hkv, L);
    size_t qp = (size_t)B * h->Hq * D * sizeof(float);
    size_t part = (size_t)B * h->Hq * p.n_split * (2 + D) * sizeof(float);
    return ((qp + 255) / 256) * 256 + part;
}

aatc_status decode_run(const aatc_calib *h, const void *q, const uint32_t *kp, const uint32_t *vp,
                       int L_cap, const int32_t *seq_lens, int L, int B, float *out, void *ws,
                       size_t ws_bytes, cudaStream_t s)
{
    if (B == 0) return AATC_OK;
    SplitPlan p = plan_splits(B, h->Hkv, L);
    float *qp = (float *)ws;
    size_t qp_bytes = (((size_t)B * h->Hq * D * sizeof(float) + 255) / 256) * 256;
    float *part = (float *)((char *)ws + qp_bytes);
    (void)ws_bytes;
    if (h->dtype == AATC_BF16)
        k_query_prep<__nv_bfloat16><<<dim3(B, h->Hq), D, 0, s>>>((const __nv_bfloat16 *)q, h->Hq, h->G,
                                                                 h->Ak32, h->tab, qp);
    else
        k_query_prep<float><<<dim3(B, h->Hq), D, 0, s>>>((const float *)q, h->Hq, h->G, h->Ak32, h->tab, qp);
    k_decode_split_simple<<<dim3(p.n_split, h->Hkv, B), DEC_TILE, 0, s>>>(
        qp, kp, vp, L_cap, seq_lens, L, h->Hkv, h->G, h->W, p.chunk, p.n_split, h->tab, part);
    k_decode_combine<<<dim3(B, h->Hq), D, 0, s>>>(part, p.n_split, h->Hq, h->G, h->tab, h->Uv32,
                                                  h->muv32, out);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

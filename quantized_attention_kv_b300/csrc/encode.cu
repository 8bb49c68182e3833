// encode.cu -- transform, quantize and bit-pack keys/values into fixed-width
// per-token records.
//
// "Attention-Aware Transform Coding Guide: KV Compression", section
// "End-to-End Implementation" (rotate into the calibrated basis, quantize each
// channel at its allocated width) and "Spend Bits Where Queries Look",
// Abstract (fixed per-token bit count).
//
// Kernels: k_encode_append (up to 16 new tokens per row, a decode step),
// k_encode_simple (fp32 inputs); bf16 prefill goes to k_encode_tc
// (encode_tc.cu).
//
// Cache tiling (per batch row and KV head, 32-token tiles of 32*W words):
// keys: token i of a tile, record word w -> half i/16 (16*W words each), row
// r = w/4 (n_r = min(4, W-4r) words, row r at 64*r), word
//     64 r + ((i%16)/2) * 2 n_r + 2 (w - 4r) + i%2;
// values: half-word e of token i -> bits 16*(i%2).. of word 16 e + i/2.
#include <cuda_bf16.h>

#include "internal.h"

namespace {

constexpr int D = AATC_D;
constexpr int ENC_TILE = 128;     // tokens per block, one thread per token

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// One block per (128-token tile, KV head, batch row x tensor).  Each thread
// owns one token: c = T x - T mu (fp32 FMA with T in shared memory),
// v = c * (1/Delta) + mid, u = clamp(rint(v), 0, 2^b - 1), then the fields of
// u are ORed into the token's record in shared memory and the record is
// written to rows start_pos + token of the packed cache.
__device__ __forceinline__ int key_word_pos(int i, int w, int W)
{
    const int r = w >> 2, nr = min(4, W - 4 * r), ii = i & 15;
    return 16 * W * (i >> 4) + 64 * r + (ii >> 1) * 2 * nr + 2 * (w - 4 * r) + (ii & 1);
}

template <typename T>
__global__ void __launch_bounds__(ENC_TILE) k_encode_simple(
    const T *__restrict__ k, const T *__restrict__ v, int L_new, int start_pos, const int32_t *row_start,
    CacheMap map, int Hkv, int Wk, int Wv, const float *__restrict__ Tk, const float *__restrict__ Tv,
    const float *__restrict__ bk, const float *__restrict__ bv, const CodecTables *__restrict__ tabs,
    const HeadPlan *__restrict__ plans, uint32_t *__restrict__ kp, uint32_t *__restrict__ vp, uint32_t *status)
{
    extern __shared__ float sm[];
    float *Ts = sm;                          // [D][D] transposed: Ts[kk][j] = T[j][kk]
    float *xs = Ts + D * D;                  // [ENC_TILE][D+1]
    uint32_t *rec = (uint32_t *)(xs + ENC_TILE * (D + 1));   // [ENC_TILE][W+1]
    __shared__ int16_t offs[D];
    const int tile = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z >> 1, tensor = blockIdx.z & 1;
    const int t = threadIdx.x;
    const int W = tensor == 0 ? Wk : Wv;   // the tensor's record words
    const T *x = (tensor == 0 ? k : v) + (((size_t)b * Hkv + h) * L_new) * D;
    const float *Tm = (tensor == 0 ? Tk : Tv) + (size_t)h * D * D;
    const float *bias = (tensor == 0 ? bk : bv) + h * D;
    const CodecTables &tb = tabs[h * 2 + tensor];
    offs[t] = plans[h * 2 + tensor].off[t];
    uint32_t *out = tensor == 0 ? kp : vp;

    for (int e = t; e < D * D; e += ENC_TILE) {
        int j = e / D, kk = e % D;
        Ts[kk * D + j] = Tm[e];
    }
    const int tok0 = tile * ENC_TILE;
    const int ntok = min(ENC_TILE, L_new - tok0);
    bool bad = false;
    for (int e = t; e < ENC_TILE * D; e += ENC_TILE) {
        int i = e / D, kk = e % D;
        float val = 0.f;
        if (i < ntok) val = to_f32(x[(size_t)(tok0 + i) * D + kk]);
        bad |= !isfinite(val);
        xs[i * (D + 1) + kk] = val;
    }
    for (int w = 0; w < W; ++w) rec[t * (W + 1) + w] = 0u;
    if (__syncthreads_or(bad) && t == 0) atomicOr(status, AATC_DEV_NONFINITE);

    const float *xr = xs + t * (D + 1);
    uint32_t *myrec = rec + t * (W + 1);
    for (int j0 = 0; j0 < D; j0 += 16) {
        float acc[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q] = 0.f;
        for (int kk = 0; kk < D; ++kk) {
            const float xv = xr[kk];
            const float4 *tr = (const float4 *)(Ts + kk * D + j0);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float4 tv = tr[q4];
                acc[4 * q4 + 0] = fmaf(tv.x, xv, acc[4 * q4 + 0]);
                acc[4 * q4 + 1] = fmaf(tv.y, xv, acc[4 * q4 + 1]);
                acc[4 * q4 + 2] = fmaf(tv.z, xv, acc[4 * q4 + 2]);
                acc[4 * q4 + 3] = fmaf(tv.w, xv, acc[4 * q4 + 3]);
            }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const int j = j0 + q;
            const int bj = tb.bits[j];
            if (bj == 0) continue;
            const float c = acc[q] - bias[j];
            float vq = fmaf(c, tb.inv_step[j], tb.mid[j]);
            vq = fminf(fmaxf(rintf(vq), 0.f), tb.top[j]);
            const uint32_t u = (uint32_t)vq;
            const int o = offs[j], sh = o & 31;
            myrec[o >> 5] |= u << sh;
            if (sh + bj > 32) myrec[(o >> 5) + 1] |= u >> (32 - sh);
        }
    }
    __syncthreads();
    // scatter the records into the tiled cache (positions row start + tok0 + i)
    const int p0 = (row_start ? row_start[b] : start_pos) + tok0;
    bool range = false;
    if (tensor == 0) {
        for (int e = t; e < ntok * W; e += ENC_TILE) {
            const int i = e / W, w = e % W, pos = p0 + i;
            const long long tw = cache_tile_word(map, b, h, Hkv, W, pos >> 5);
            if (tw < 0) { range = true; continue; }
            out[tw + key_word_pos(pos & 31, w, W)] = rec[i * (W + 1) + w];
        }
    } else {
        uint16_t *out16 = (uint16_t *)out;
        for (int e = t; e < ntok * 2 * W; e += ENC_TILE) {
            const int i = e / (2 * W), q = e % (2 * W), pos = p0 + i;
            const long long tw = cache_tile_word(map, b, h, Hkv, W, pos >> 5);
            if (tw < 0) { range = true; continue; }
            const uint32_t wv = rec[i * (W + 1) + (q >> 1)];
            const long long word = tw + 16 * q + ((pos & 31) >> 1);
            out16[2 * word + (pos & 1)] = (uint16_t)(wv >> (16 * (q & 1)));
        }
    }
    if (range) atomicOr(status, AATC_DEV_RANGE);
}

// Append path: a few new tokens per row, as in a decode step.  One CTA of
// D threads per (KV head, tensor, batch row); thread j owns coefficient j and
// computes it exactly as k_encode_simple does (fp32 FMA over k = 0..127,
// minus T mu, scaled, rounded half to even, clamped).  The codes are ORed into
// the token's record in shared memory and the record goes to its place in the
// tiled cache.  T (64 KB, read from the handle) is staged in shared memory by
// cp.async before the kernel waits for its predecessor on the stream
// (programmatic dependent launch), so that copy overlaps the previous kernel;
// the new tokens are read and the cache written only after the wait.
constexpr int APPEND_MAX = 16;    // tokens per row served by this path
constexpr int TPAD = D + 4;       // floats per staged row of T (16-byte rows, conflict-free float4 reads)
constexpr int MAX_W = 8 * D / 32; // record words at 8 bits per channel

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(D) k_encode_append(
    const T *__restrict__ k, const T *__restrict__ v, int L_new, int start_pos, const int32_t *row_start,
    CacheMap map, int Hkv, int Wk, int Wv, const float *__restrict__ Tk, const float *__restrict__ Tv, const float *__restrict__ bk,
    const float *__restrict__ bv, const CodecTables *__restrict__ tabs, const HeadPlan *__restrict__ plans,
    uint32_t *__restrict__ kp, uint32_t *__restrict__ vp, uint32_t *status)
{
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ __align__(16) float Ts[];   // [D][TPAD]: row j of T
    __shared__ float xs[D];
    __shared__ uint32_t rec[MAX_W];
    const int h = blockIdx.x, tensor = blockIdx.y, b = blockIdx.z, j = threadIdx.x;
    const int ht = h * 2 + tensor;
    const int W = tensor == 0 ? Wk : Wv;   // the tensor's record words

    // handle data only, ahead of the wait
    const float4 *src = reinterpret_cast<const float4 *>((tensor == 0 ? Tk : Tv) + (size_t)h * D * D);
#pragma unroll 8
    for (int i = 0; i < D * D / 4 / D; ++i) {
        const int e4 = j + i * D;   // float4 e4 of T: row e4 / 32, columns 4 (e4 % 32) ..
        cp_async16(&Ts[(e4 >> 5) * TPAD + (e4 & 31) * 4], src + e4);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    const float bias = (tensor == 0 ? bk : bv)[h * D + j];
    const float inv = tabs[ht].inv_step[j], mid = tabs[ht].mid[j], top = tabs[ht].top[j];
    const int bits = tabs[ht].bits[j], off = plans[ht].off[j];
    asm volatile("cp.async.wait_all;" ::: "memory");

    // the new tokens and the cache may belong to the previous kernel on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const T *x = (tensor == 0 ? k : v) + ((size_t)b * Hkv + h) * L_new * D;
    uint32_t *out = tensor == 0 ? kp : vp;
    const int pos0 = row_start ? row_start[b] : start_pos;
    bool bad = false, range = false;
    for (int n = 0; n < L_new; ++n) {
        const float xv = to_f32(x[(size_t)n * D + j]);
        bad |= !isfinite(xv);
        xs[j] = xv;
        if (j < W) rec[j] = 0u;
        __syncthreads();   // xs, rec, and (first token) every thread's staged rows of T
        const float4 *tr = reinterpret_cast<const float4 *>(&Ts[j * TPAD]);
        float acc = 0.f;
#pragma unroll 8
        for (int k4 = 0; k4 < D / 4; ++k4) {
            const float4 t = tr[k4];
            acc = fmaf(t.x, xs[4 * k4 + 0], acc);
            acc = fmaf(t.y, xs[4 * k4 + 1], acc);
            acc = fmaf(t.z, xs[4 * k4 + 2], acc);
            acc = fmaf(t.w, xs[4 * k4 + 3], acc);
        }
        if (bits > 0) {
            float vq = fmaf(acc - bias, inv, mid);
            vq = fminf(fmaxf(rintf(vq), 0.f), top);
            const uint32_t u = (uint32_t)vq;
            const int sh = off & 31;
            atomicOr(&rec[off >> 5], u << sh);
            if (sh + bits > 32) atomicOr(&rec[(off >> 5) + 1], u >> (32 - sh));
        }
        __syncthreads();
        const int pos = pos0 + n;
        if (j < (tensor == 0 ? W : 2 * W)) {
            const long long tw = cache_tile_word(map, b, h, Hkv, W, pos >> 5);
            if (tw < 0) {
                range = true;
            } else if (tensor == 0) {
                out[tw + key_word_pos(pos & 31, j, W)] = rec[j];
            } else {
                const long long word = tw + 16 * j + ((pos & 31) >> 1);
                reinterpret_cast<uint16_t *>(out)[2 * word + (pos & 1)] = (uint16_t)(rec[j >> 1] >> (16 * (j & 1)));
            }
        }
        __syncthreads();   // xs and rec are reused by the next token
    }
    if (__syncthreads_or(bad) && j == 0) atomicOr(status, AATC_DEV_NONFINITE);
    if (range) atomicOr(status, AATC_DEV_RANGE);
}

template <typename T>
aatc_status launch_append(const aatc_calib *h, const void *k, const void *v, int B, int L_new, int start_pos,
                          const int32_t *row_start, const CacheMap &map, uint32_t *kp, uint32_t *vp, cudaStream_t s)
{
    static const size_t smem = (size_t)D * TPAD * sizeof(float);
    auto kern = k_encode_append<T>;
    aatc_status st = kernel_smem_limit((const void *)kern, smem);
    if (st != AATC_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(h->Hkv, 2, B);
    cfg.blockDim = dim3(D);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    AATC_CUDA(cudaLaunchKernelEx(&cfg, kern, (const T *)k, (const T *)v, L_new, start_pos, row_start, map, h->Hkv, h->Wk, h->Wv,
                                 (const float *)h->Tk32, (const float *)h->Tv32, (const float *)h->bk32,
                                 (const float *)h->bv32, (const CodecTables *)h->tab, (const HeadPlan *)h->plan,
                                 kp, vp, h->status));
    return AATC_OK;
}

}  // namespace

aatc_status encode_run(const aatc_calib *h, const void *k, const void *v, int B, int L_new, int start_pos,
                       const int32_t *row_start, const CacheMap &map, uint32_t *kp, uint32_t *vp, cudaStream_t s)
{
    if (L_new == 0 || B == 0) return AATC_OK;
    if (L_new <= APPEND_MAX && B <= 65535) {   // a decode step's new tokens
        if (h->dtype == AATC_BF16)
            return launch_append<__nv_bfloat16>(h, k, v, B, L_new, start_pos, row_start, map, kp, vp, s);
        return launch_append<float>(h, k, v, B, L_new, start_pos, row_start, map, kp, vp, s);
    }
    if (h->dtype == AATC_BF16 && h->tmap_ok && h->Wk <= 16 && h->Wv <= 16)
        return encode_tc_run(h, k, v, B, L_new, start_pos, row_start, map, kp, vp, s);
    const size_t smem = (size_t)D * D * 4 + (size_t)ENC_TILE * (D + 1) * 4 +
                        (size_t)ENC_TILE * ((h->Wk > h->Wv ? h->Wk : h->Wv) + 1) * 4;
    const dim3 grid((L_new + ENC_TILE - 1) / ENC_TILE, h->Hkv, 2 * B);
    if (h->dtype == AATC_BF16) {
        auto kern = k_encode_simple<__nv_bfloat16>;
        aatc_status st = kernel_smem_limit((const void *)kern, smem);
        if (st != AATC_OK) return st;
        kern<<<grid, ENC_TILE, smem, s>>>((const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, L_new,
                                          start_pos, row_start, map, h->Hkv, h->Wk, h->Wv, h->Tk32, h->Tv32, h->bk32,
                                          h->bv32, h->tab, h->plan, kp, vp, h->status);
    } else {
        auto kern = k_encode_simple<float>;
        aatc_status st = kernel_smem_limit((const void *)kern, smem);
        if (st != AATC_OK) return st;
        kern<<<grid, ENC_TILE, smem, s>>>((const float *)k, (const float *)v, L_new, start_pos, row_start, map,
                                          h->Hkv, h->Wk, h->Wv, h->Tk32, h->Tv32, h->bk32, h->bv32, h->tab, h->plan,
                                          kp, vp, h->status);
    }
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

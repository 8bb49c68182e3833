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
// each packed record is streamed once.
//
// Fast path (record words <= 16, at most 4 code pieces per record byte):
//   k_qprep_fast   per (batch row, KV head, head group): q' for the group's
//                  query heads, expanded to one fp16 hi/lo weight per record
//                  piece in mma.sync B-fragment order; zeroes the merge ticket.
//   k_decode_fast  per (split, KV head, batch row x head group): 4 warps, each
//                  streaming its own 32-token tiles into shared memory with
//                  cp.async.bulk, unpacking pieces with one AND per two fp16
//                  operands, scores and P.V on mma.sync (fp16 hi/lo operands,
//                  fp32 accumulation), online softmax in exp2 form.  Warps and
//                  splits merge by log-sum-exp; the last CTA of a (batch row,
//                  KV head, head group) applies Uv and writes the output.
// General path (any shape): one thread per token, codes read by offset.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "internal.h"

namespace {

constexpr int D = AATC_D;
constexpr int TILE = 32;
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

int sm_count()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            n = 148;
    }
    return n;
}

// =============================================================== fast path
constexpr int FSTAGES = 3;       // tiles in flight per warp
constexpr int PSTRIDE = 40;      // halfs per row of the per-warp P buffer (32 tokens + pad)
constexpr int FAST_MAX_W = 16;
constexpr int PROW = 4 + D;      // floats per partial: m, l, 2 pad, acc[D] (acc 16-byte aligned)
constexpr size_t FINAL_SMEM = (size_t)D * D * 4 + 2 * 8 * D * 4;   // Uv^T + channel sums + cbar

// Work split: every (batch row, KV head, head group) is a "unit" of
// n_tiles = ceil(L/32) tiles.  The units' tiles are laid end to end and
// cut into C equal contiguous ranges, one per CTA (C = resident CTAs), so
// the load is balanced whatever the batch.  A CTA works through the units
// its range touches one "segment" at a time and leaves one partial per
// segment; CTA c covers unit u iff its range meets the unit's tiles, and
// the CTA holding global tile x is c(x) = ((x + 1) C - 1) / T.
struct FastGeom {
    int NT;          // 8-column n-tiles (each: 4 query heads x hi/lo)
    int HPG;         // query heads per head group (4 NT)
    int HG;          // head groups per KV head
    int FW;          // warps per CTA
    int rows;        // key rows of 4 record words
    int groups;      // value groups of 8 half-words
    int ksteps;      // 4 rows
    int n_tiles;     // tiles per unit
    int units;       // B * Hkv * HG
    int C;           // CTAs
    int PMAX;        // partial slots per unit
    size_t stage_bytes, smem, qtab_words, ws_qtab, ws_qsc, ws_part, ws_cnt, ws_total;
};

__host__ __device__ __forceinline__ int cta_of_tile(long long x, int C, long long T)
{
    return (int)(((x + 1) * C - 1) / T);
}

size_t fast_smem(int FW, int W, int groups, int HPG, int NT, int ksteps, int rows)
{
    const size_t SB = 256 * (size_t)W + 512;
    const size_t rows_tot = 64 * (size_t)groups;
    const size_t merge = (size_t)FW * (rows_tot + 2) * HPG * 4 + (size_t)D * HPG * 4;
    size_t big = (size_t)FW * FSTAGES * SB;
    big = big > merge ? big : merge;
    big = big > FINAL_SMEM ? big : FINAL_SMEM;
    big = (big + 127) & ~(size_t)127;
    return big + (size_t)FW * FSTAGES * 8 + (size_t)FW * 16 * PSTRIDE * 2 + (size_t)ksteps * NT * 32 * 8 +
           (size_t)rows * 4 * 8 * 4 + (size_t)groups * 64 * 4 + 256 * 2 + 8 * 4 + 16;
}

template <int GMAX, int NT, int FW> __global__ void k_decode_fast(struct FastArgs a);

int fast_ctas_per_sm(int groups, int NT, int FW, size_t smem);

FastGeom fast_geom(const aatc_calib *h, int B, int L)
{
    FastGeom f;
    f.NT = h->G <= 4 ? 1 : 2;
    f.HPG = 4 * f.NT;
    f.HG = (h->G + f.HPG - 1) / f.HPG;
    f.FW = f.NT == 1 ? 12 : 8;
    f.rows = (h->W + 3) / 4;
    f.groups = (2 * h->W + 7) / 8;
    f.ksteps = 4 * f.rows;
    f.n_tiles = L > 0 ? (L + TILE - 1) / TILE : 0;
    f.units = B * h->Hkv * f.HG;
    f.smem = fast_smem(f.FW, h->W, f.groups, f.HPG, f.NT, f.ksteps, f.rows);
    const int per_sm = fast_ctas_per_sm(f.groups, f.NT, f.FW, f.smem);
    const long long T = (long long)f.units * f.n_tiles;
    long long C = (long long)sm_count() * per_sm;
    if (C > T) C = T > 0 ? T : 1;
    f.C = (int)C;
    f.PMAX = (int)((f.C + f.units - 1) / f.units) + 1;
    f.stage_bytes = 256 * (size_t)h->W + 512;
    f.qtab_words = (size_t)f.ksteps * f.NT * 32 * 2;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t uz = (size_t)f.units;
    f.ws_qtab = up(uz * f.qtab_words * 4);
    f.ws_qsc = up(uz * 8 * 4);
    f.ws_part = up(uz * f.PMAX * f.HPG * PROW * 4);
    f.ws_cnt = up(uz * 4);
    f.ws_total = f.ws_qtab + f.ws_qsc + f.ws_part + f.ws_cnt;
    return f;
}

bool fast_ok(const aatc_calib *h) { return h->W <= FAST_MAX_W && h->fast_layout; }

// ---- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *mb, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mb)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive_expect(uint64_t *mb, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(mb)), "r"(bytes)
                 : "memory");
}

// Bounded wait of a whole warp on a phase of an mbarrier: false (on every
// lane) if it did not complete within the iteration limit.
__device__ __forceinline__ bool mbar_wait(uint64_t *mb, uint32_t parity)
{
    const uint32_t a = smem_u32(mb);
    for (int it = 0; it < (1 << 22); ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (__all_sync(0xffffffffu, done)) return true;
    }
    return false;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *mb)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(mb))
        : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

struct FastArgs {
    const uint32_t *kp, *vp;
    const int32_t *seq_lens;
    int L, L_cap, W, rows, groups, Hkv, G, HG, HPG, n_tiles, units, C, PMAX;
    const HeadPlan *plan;
    const uint32_t *qtab;   // [units][ksteps][NT][32] uint2
    const float *qsc;       // [units][8]
    float *part;            // [units][PMAX][HPG][PROW]
    uint32_t *cnt;          // [units]
    const CodecTables *tab;
    const float *UvT, *muv;
    float *out;
    uint32_t *status;
};

// q' of the head group's query heads, expanded to per-piece fp16 hi/lo
// weights in B-fragment order: entry (kstep, n-tile t, lane) = (b0, b1) with
// column n = 8t + lane/4 = (head n/2, hi if n even else lo), rows of k-step
// (r, s) from record word 4r + lane%4, slots 2s (b0) and 2s+1 (b1), low half
// first.  Weight of a piece = q'_ch * 2^ex * S, S a power of two per head
// keeping every weight below 2^13; qsc[head] = 2^24 / S * log2(e) turns the
// accumulated score back into log2 units.  Also zeroes the unit's merge
// ticket and pulls the unit's Uv^T into L2 for the final merge.
// One block of 256 threads per unit; A_k^T arrives in shared memory by one
// bulk copy, thread j (+128) sums half of its rows for channel j.
constexpr int QP_THREADS = 2 * D;
constexpr size_t QP_SMEM = (size_t)D * D * 4 + 16;
template <typename T>
__global__ void __launch_bounds__(QP_THREADS) k_qprep_fast(
    const T *__restrict__ q, const float *__restrict__ AkT, const float *__restrict__ UvT,
    const CodecTables *__restrict__ tabs, const HeadPlan *__restrict__ plans, int Hkv, int G, int HG, int HPG,
    int NT, int ksteps, uint32_t *__restrict__ qtab, float *__restrict__ qsc, uint32_t *__restrict__ cnt,
    uint32_t *status)
{
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ __align__(128) unsigned char qsm[];
    float *As = reinterpret_cast<float *>(qsm);          // [D][D] = AkT of this head
    __shared__ float qs[8][D];
    __shared__ float pa[2][8][D];
    __shared__ float S[8];
    __shared__ int16_t slot_s[AATC_PLAN_SLOTS / 2][8][2];   // key words 0..15: ch | (ex + 64) << 8
    __shared__ __align__(8) uint64_t bar;
    const int b = blockIdx.x, h = blockIdx.y, hg = blockIdx.z, tid = threadIdx.x;
    const int j = tid & (D - 1), kh = tid >> 7;
    const int unit = (b * Hkv + h) * HG + hg;
    const int Hq = Hkv * G;
    if (tid == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect(&bar, D * D * 4);
        bulk_g2s(As, AkT + (size_t)h * D * D, D * D * 4, &bar);
        if (hg == 0 && b == 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(UvT + (size_t)h * D * D), "r"(D * D * 4)
                         : "memory");
        cnt[unit] = 0u;
    }
    for (int e = tid; e < 8 * D; e += QP_THREADS) {
        const int i = e >> 7, cc = e & (D - 1), gi = hg * HPG + i;
        qs[i][cc] = (i < HPG && gi < G) ? to_f32(q[((size_t)b * Hq + h * G + gi) * D + cc]) : 0.f;
    }
    const HeadPlan &pk = plans[h * 2 + 0];
    for (int e = tid; e < (AATC_PLAN_SLOTS / 2) * 16; e += QP_THREADS) {
        const int w = e >> 4, k = (e >> 1) & 7, half = e & 1;
        const int ch = pk.ch[w][k][half];
        slot_s[w][k][half] = (int16_t)(ch < 0 ? -1 : (ch | ((pk.ex[w][k][half] + 64) << 8)));
    }
    __syncthreads();
    if (!mbar_wait(&bar, 0)) {
        if (tid == 0) atomicOr(status, AATC_DEV_TIMEOUT);
        return;
    }
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 4
    for (int k = kh * 64; k < kh * 64 + 64; ++k) {
        const float av = As[k * D + j];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(av, qs[i][k], acc[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) pa[kh][i][j] = acc[i];
    __syncthreads();
    const CodecTables &tk = tabs[h * 2 + 0];
    if (tid < D) {
        const float scale = tk.bits[j] ? tk.step[j] * 0.08838834764831845f : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) pa[0][i][j] = (pa[0][i][j] + pa[1][i][j]) * scale;
    }
    __syncthreads();
    {   // warp i: largest |q'| of head i
        const int wi = tid >> 5, ln = tid & 31;
        if (wi < HPG) {
            float mx = 0.f;
            for (int k = ln; k < D; k += 32) mx = fmaxf(mx, fabsf(pa[0][wi][k]));
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (ln == 0) {
                // pieces carry 2^ex with ex <= 7: keep mx * 2^7 * S below 2^13
                int e = 0;
                if (mx > 0.f) frexpf(mx, &e);
                S[wi] = mx > 0.f ? ldexpf(1.f, 6 - e) : 1.f;
                qsc[unit * 8 + wi] = ldexpf(1.f, 24) / S[wi] * LOG2E;
            }
        }
    }
    __syncthreads();
    const int entries = ksteps * NT * 32;
    uint2 *dst = reinterpret_cast<uint2 *>(qtab) + (size_t)unit * entries;
    for (int en = tid; en < entries; en += QP_THREADS) {
        const int lane = en & 31, t = (en >> 5) % NT, ks = (en >> 5) / NT;
        const int r = ks >> 2, s4 = ks & 3;
        const int n = 8 * t + (lane >> 2), i = n >> 1, part = n & 1;
        const int w = 4 * r + (lane & 3);
        uint32_t o2[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int k = 2 * s4 + rr;
            float v2[2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int sl = slot_s[w][k][half];
                float val = 0.f;
                if (sl >= 0 && hg * HPG + i < G) val = ldexpf(pa[0][i][sl & 255] * S[i], (sl >> 8) - 64);
                const float hi = __half2float(__float2half_rn(val));
                v2[half] = part ? val - hi : hi;
            }
            o2[rr] = pack_half2(v2[0], v2[1]);
        }
        dst[en] = make_uint2(o2[0], o2[1]);
    }
}

template <int GMAX, int NT, int FW>
__global__ void __launch_bounds__(FW * 32) k_decode_fast(FastArgs a)
{
    constexpr int NTH = FW * 32;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int g = lane >> 2, c = lane & 3;
    const int W = a.W, rows = a.rows, groups = a.groups, HPG = a.HPG;
    const int ksteps = rows * 4;

    // shared memory carve-up (sizes as in fast_smem)
    const size_t SB = 256 * (size_t)W + 512;
    const size_t rows_tot = 64 * (size_t)groups;
    const size_t merge = (size_t)FW * (rows_tot + 2) * HPG * 4 + (size_t)D * HPG * 4;
    size_t big = (size_t)FW * FSTAGES * SB;
    big = big > merge ? big : merge;
    big = big > FINAL_SMEM ? big : FINAL_SMEM;
    big = (big + 127) & ~(size_t)127;
    unsigned char *stage_base = smem;
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + big);
    __half *pbuf = reinterpret_cast<__half *>(mbar + FW * FSTAGES);
    uint2 *qtab_s = reinterpret_cast<uint2 *>(pbuf + FW * 16 * PSTRIDE);
    uint32_t *kmask_s = reinterpret_cast<uint32_t *>(qtab_s + ksteps * NT * 32);
    uint32_t *vmask_s = kmask_s + rows * 4 * 8;
    int16_t *vrow_s = reinterpret_cast<int16_t *>(vmask_s + groups * 64);   // [groups*64] (ch << 8 | ex + 64)
    float *sc_s = reinterpret_cast<float *>(vrow_s + 256);
    __shared__ int s_last;
    __shared__ float red[NTH];
    __shared__ float cm[8], cl[8], cs[8][FW];
    __shared__ __align__(8) uint64_t ubar;     // Uv^T bulk copy of the final merge
    __shared__ float vmid_s[256];              // value piece midpoints (2^w-1)/2 * 2^(p-24), per row

    uint64_t *my_mbar = mbar + warp * FSTAGES;
    unsigned char *my_stage = stage_base + (size_t)warp * FSTAGES * SB;
    const uint32_t tile_bytes = 128u * W;
    if (lane == 0) {
        for (int s = 0; s < FSTAGES; ++s) mbar_init(&my_mbar[s], 1);
        if (warp == 0) mbar_init(&ubar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    int n_final = 0;   // final merges done by this CTA (phases of ubar)
    // The warp's n-th tile (over all its segments) goes through stage n % FSTAGES
    // and completes phase n / FSTAGES of that stage's barrier.
    int n_issued = 0, n_done = 0;

    const long long T = (long long)a.units * a.n_tiles;
    const long long lo = (long long)blockIdx.x * T / a.C, hi = (long long)(blockIdx.x + 1) * T / a.C;
    bool waited = false;
    for (long long x = lo; x < hi;) {
        // ---- next segment: unit u, tiles [ta, tb) of the unit
        const int u = (int)(x / a.n_tiles);
        const int ta = (int)(x - (long long)u * a.n_tiles);
        const long long uend = (long long)(u + 1) * a.n_tiles;
        const int tb = (int)((hi < uend ? hi : uend) - (long long)u * a.n_tiles);
        x = (long long)u * a.n_tiles + tb;
        const int b = u / (a.Hkv * a.HG), h = (u / a.HG) % a.Hkv, hg = u % a.HG;
        const int len = a.seq_lens ? min(max(a.seq_lens[b], 0), a.L) : a.L;
        const int t0 = ta, t1 = min(tb, (len + TILE - 1) / TILE);
        const size_t slab = ((size_t)b * a.Hkv + h) * (size_t)a.L_cap * W;

        auto issue = [&](int tile, int s) {
            unsigned char *dst = my_stage + s * SB;
            mbar_arrive_expect(&my_mbar[s], 2 * tile_bytes);
            bulk_g2s(dst, a.kp + slab + (size_t)tile * TILE * W, tile_bytes, &my_mbar[s]);
            bulk_g2s(dst + tile_bytes, a.vp + slab + (size_t)tile * TILE * W, tile_bytes, &my_mbar[s]);
        };
        for (int i = 0; i < FSTAGES; ++i) {
            const int tile = t0 + warp + i * FW;
            if (tile < t1) {
                if (lane == 0) issue(tile, n_issued % FSTAGES);
                ++n_issued;
            }
        }

        // tables of this unit
        const HeadPlan &pk = a.plan[h * 2 + 0];
        const HeadPlan &pv = a.plan[h * 2 + 1];
        for (int e = tid; e < rows * 4 * 8; e += NTH) kmask_s[e] = pk.mask[e >> 3][e & 7];
        for (int e = tid; e < groups * 64; e += NTH) vmask_s[e] = pv.mask[e >> 3][e & 7];
        for (int e = tid; e < groups * 64; e += NTH) {
            // row e = (group, m4, rr): half-word 8 group + rr%8, slot 2 m4 + rr/8
            const int gr = e >> 6, m4 = (e >> 4) & 3, rr = e & 15;
            const int hw = 8 * gr + (rr & 7), k = 2 * m4 + (rr >> 3);
            const int ch = pv.ch[hw][k][0];
            vrow_s[e] = (int16_t)(ch < 0 ? -1 : (ch << 8) | (pv.ex[hw][k][0] + 64));
            // the mask holds (2^w - 1) << p in each half: its low half / 2 is the
            // piece's midpoint times 2^p
            vmid_s[e] = ldexpf((float)(pv.mask[hw][k] & 0xFFFFu), -25);
        }
        if (!waited) {   // query weights and tickets come from k_qprep_fast
            asm volatile("griddepcontrol.wait;" ::: "memory");
            waited = true;
        }
        {
            const uint2 *src = reinterpret_cast<const uint2 *>(a.qtab) + (size_t)u * ksteps * NT * 32;
            for (int e = tid; e < ksteps * NT * 32; e += NTH) qtab_s[e] = src[e];
            if (tid < 8) sc_s[tid] = a.qsc[u * 8 + tid];
        }
        __syncthreads();

        float m_run[NT], l_run[NT], sc[NT];
        float acc[GMAX][4][NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            m_run[t] = -INFINITY;
            l_run[t] = 0.f;
            sc[t] = sc_s[4 * t + c];
        }
#pragma unroll
        for (int gr = 0; gr < GMAX; ++gr)
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4)
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[gr][m4][t][k] = 0.f;

        __half *pw = pbuf + warp * 16 * PSTRIDE;
        bool failed = false;
        for (int it = 0;; ++it) {
            const int tile = t0 + warp + it * FW;
            if (tile >= t1) break;
            const int s = n_done % FSTAGES;
            if (!mbar_wait(&my_mbar[s], (uint32_t)((n_done / FSTAGES) & 1))) {
                failed = true;
                break;
            }
            ++n_done;
            const uint32_t *Kt = reinterpret_cast<const uint32_t *>(my_stage + s * SB);
            const uint32_t *Vt = Kt + TILE * W;

            // ---- scores: rows = tokens (row g: 2g, row g+8: 2g+1 of the half), k = record pieces
            float C[2][NT][4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int k = 0; k < 4; ++k) C[hf][t][k] = 0.f;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r >= rows) break;
                    const int nr = min(4, W - 4 * r);
                    const uint2 kw =
                        *reinterpret_cast<const uint2 *>(Kt + hf * 16 * W + 64 * r + g * 2 * nr + 2 * c);
                    const uint4 mA = *reinterpret_cast<const uint4 *>(kmask_s + (4 * r + c) * 8);
                    const uint4 mB = *reinterpret_cast<const uint4 *>(kmask_s + (4 * r + c) * 8 + 4);
                    const uint32_t mk[8] = {mA.x, mA.y, mA.z, mA.w, mB.x, mB.y, mB.z, mB.w};
                    const uint32_t x0 = kw.x, x1 = kw.y, y0 = x0 >> 8, y1 = x1 >> 8;
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        const uint32_t sa = s4 < 2 ? x0 : y0, sb = s4 < 2 ? x1 : y1;
                        const uint32_t A0 = sa & mk[2 * s4], A1 = sb & mk[2 * s4];
                        const uint32_t A2 = sa & mk[2 * s4 + 1], A3 = sb & mk[2 * s4 + 1];
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            const uint2 bq = qtab_s[((r * 4 + s4) * NT + t) * 32 + lane];
                            mma16816(C[hf][t], A0, A1, A2, A3, bq.x, bq.y);
                        }
                    }
                }
            }

            // ---- online softmax (log2 domain); thread owns head 4t+c of tokens 16hf+2g, +1
            const int tb0 = tile * TILE;
            float psh[NT], psl[NT];   // this tile's sums of the fp16 P operands (hi, lo) per head
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float z[2][2];
                float mt = -INFINITY;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int tau = tb0 + 16 * hf + 2 * g;
                    z[hf][0] = tau < len ? (C[hf][t][0] + C[hf][t][1]) * sc[t] : -INFINITY;
                    z[hf][1] = tau + 1 < len ? (C[hf][t][2] + C[hf][t][3]) * sc[t] : -INFINITY;
                    mt = fmaxf(mt, fmaxf(z[hf][0], z[hf][1]));
                }
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
                const float mn = fmaxf(m_run[t], mt);
                const float alpha = (mn == -INFINITY) ? 1.f : exp2f(m_run[t] - mn);
                m_run[t] = mn;
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    l_run[t] *= alpha;
#pragma unroll
                    for (int gr = 0; gr < GMAX; ++gr)
#pragma unroll
                        for (int m4 = 0; m4 < 4; ++m4)
#pragma unroll
                            for (int k = 0; k < 4; ++k) acc[gr][m4][t][k] *= alpha;
                }
                psh[t] = 0.f;
                psl[t] = 0.f;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float p0 = z[hf][0] == -INFINITY ? 0.f : exp2f(z[hf][0] - mn);
                    const float p1 = z[hf][1] == -INFINITY ? 0.f : exp2f(z[hf][1] - mn);
                    l_run[t] += p0 + p1;
                    // P scaled by 2^14: hi/lo fp16 pair per token (hi in column 2c, lo in 2c+1)
                    const float s0 = p0 * 16384.f, s1 = p1 * 16384.f;
                    const __half2 hi2 = __floats2half2_rn(s0, s1);
                    const float2 hif = __half22float2(hi2);
                    const __half2 lo2 = __floats2half2_rn(s0 - hif.x, s1 - hif.y);
                    const float2 lof = __half22float2(lo2);
                    psh[t] += hif.x + hif.y;
                    psl[t] += lof.x + lof.y;
                    const int tau = 16 * hf + 2 * g;
                    *reinterpret_cast<__half2 *>(pw + (8 * t + 2 * c) * PSTRIDE + tau) = hi2;
                    *reinterpret_cast<__half2 *>(pw + (8 * t + 2 * c + 1) * PSTRIDE + tau) = lo2;
                }
            }
            __syncwarp();
#pragma unroll
            for (int t = 0; t < NT; ++t) {
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    psh[t] += __shfl_xor_sync(0xffffffffu, psh[t], o);
                    psl[t] += __shfl_xor_sync(0xffffffffu, psl[t], o);
                }
            }

            // ---- P.V: rows = value pieces (half-word 8 gr + g, slot 2 m4 / 2 m4 + 1), k = tokens
            uint2 bp[2][NT];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    bp[kk][t] = *reinterpret_cast<const uint2 *>(pw + (8 * t + g) * PSTRIDE + 8 * c + 4 * kk);
#pragma unroll
            for (int gr = 0; gr < GMAX; ++gr) {
                if (gr >= groups) break;
                const int e = 8 * gr + g;
                const uint4 pq = *reinterpret_cast<const uint4 *>(Vt + e * 16 + 4 * c);
                const uint4 mA = *reinterpret_cast<const uint4 *>(vmask_s + e * 8);
                const uint4 mB = *reinterpret_cast<const uint4 *>(vmask_s + e * 8 + 4);
                const uint32_t mv[8] = {mA.x, mA.y, mA.z, mA.w, mB.x, mB.y, mB.z, mB.w};
                const uint32_t xs[4] = {pq.x, pq.y, pq.z, pq.w};
                const uint32_t ys[4] = {pq.x >> 8, pq.y >> 8, pq.z >> 8, pq.w >> 8};
#pragma unroll
                for (int m4 = 0; m4 < 4; ++m4) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint32_t u0 = m4 < 2 ? xs[2 * kk] : ys[2 * kk];
                        const uint32_t u1 = m4 < 2 ? xs[2 * kk + 1] : ys[2 * kk + 1];
                        const uint32_t A0 = u0 & mv[2 * m4], A1 = u0 & mv[2 * m4 + 1];
                        const uint32_t A2 = u1 & mv[2 * m4], A3 = u1 & mv[2 * m4 + 1];
#pragma unroll
                        for (int t = 0; t < NT; ++t)
                            mma16816(acc[gr][m4][t], A0, A1, A2, A3, bp[kk][t].x, bp[kk][t].y);
                    }
                    // keep the sums centred: subtract each piece's midpoint times the
                    // tile's P mass, so the tensor-core accumulation (which does not
                    // round to nearest) only ever carries small values
                    const float c0 = vmid_s[(gr * 4 + m4) * 16 + g], c1 = vmid_s[(gr * 4 + m4) * 16 + g + 8];
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        acc[gr][m4][t][0] = fmaf(-c0, psh[t], acc[gr][m4][t][0]);
                        acc[gr][m4][t][1] = fmaf(-c0, psl[t], acc[gr][m4][t][1]);
                        acc[gr][m4][t][2] = fmaf(-c1, psh[t], acc[gr][m4][t][2]);
                        acc[gr][m4][t][3] = fmaf(-c1, psl[t], acc[gr][m4][t][3]);
                    }
                }
            }
            __syncwarp();
            const int nt = tile + FSTAGES * FW;
            if (nt < t1) {
                if (lane == 0) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(nt, n_issued % FSTAGES);
                }
                ++n_issued;
            }
        }
        if (failed) {
            if (lane == 0) atomicOr(a.status, AATC_DEV_TIMEOUT);
            // let copies still in flight land before the shared memory is reused
            for (; n_done < n_issued; ++n_done)
                mbar_wait(&my_mbar[n_done % FSTAGES], (uint32_t)((n_done / FSTAGES) & 1));
#pragma unroll
            for (int t = 0; t < NT; ++t) { m_run[t] = -INFINITY; l_run[t] = 0.f; }
        }

        // ---- warp partials -> shared memory (the stage area is free now)
        __syncthreads();
        float *wm = reinterpret_cast<float *>(stage_base);          // [FW][HPG]
        float *wl = wm + FW * HPG;                                   // [FW][HPG]
        float *wacc = wl + FW * HPG;                                 // [FW][rows_tot][HPG]
        float *ach = wacc + (size_t)FW * rows_tot * HPG;             // [D][HPG]
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float l = l_run[t];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            const int i = 4 * t + c;
            if (g == 0) {
                wm[warp * HPG + i] = m_run[t];
                wl[warp * HPG + i] = l;
            }
#pragma unroll
            for (int gr = 0; gr < GMAX; ++gr) {
                if (gr >= groups) break;
#pragma unroll
                for (int m4 = 0; m4 < 4; ++m4) {
                    const int row = (gr * 4 + m4) * 16 + g;
                    float *dst = wacc + ((size_t)warp * rows_tot + row) * HPG + i;
                    dst[0] = failed ? 0.f : acc[gr][m4][t][0] + acc[gr][m4][t][1];
                    dst[8 * HPG] = failed ? 0.f : acc[gr][m4][t][2] + acc[gr][m4][t][3];
                }
            }
        }
        for (int e = tid; e < D * HPG; e += NTH) ach[e] = 0.f;
        __syncthreads();

        // ---- merge the warps, map pieces to channels: sum_i p_i u_ij (p unscaled)
        if (tid < HPG) {
            const int i = tid;
            float M = -INFINITY;
            for (int w = 0; w < FW; ++w) M = fmaxf(M, wm[w * HPG + i]);
            float Ls = 0.f;
            for (int w = 0; w < FW; ++w) {
                const float f = (M == -INFINITY || wm[w * HPG + i] == -INFINITY) ? 0.f : exp2f(wm[w * HPG + i] - M);
                cs[i][w] = f;
                Ls += wl[w * HPG + i] * f;
            }
            cm[i] = M;
            cl[i] = Ls;
        }
        __syncthreads();
        for (int e = tid; e < (int)rows_tot * HPG; e += NTH) {
            const int row = e / HPG, i = e % HPG;
            const int rv = vrow_s[row];
            if (rv < 0) continue;
            float v = 0.f;
#pragma unroll 4
            for (int w = 0; w < FW; ++w) v = fmaf(wacc[((size_t)w * rows_tot + row) * HPG + i], cs[i][w], v);
            // fp16 operands: piece value * 2^(p-24) and P * 2^14; piece * 2^ex is the code part
            atomicAdd(&ach[(rv >> 8) * HPG + i], ldexpf(v, (rv & 255) - 64 + 10));
        }
        __syncthreads();
        const int c_first = cta_of_tile((long long)u * a.n_tiles, a.C, T);
        const int c_last = cta_of_tile((long long)(u + 1) * a.n_tiles - 1, a.C, T);
        const int slot = blockIdx.x - c_first;
        {
            float *P = a.part + ((size_t)u * a.PMAX + slot) * HPG * PROW;
            for (int e = tid; e < HPG * PROW; e += NTH) {
                const int i = e / PROW, j = e % PROW;
                P[e] = j == 0 ? cm[i] : (j == 1 ? cl[i] : (j < 4 ? 0.f : ach[(j - 4) * HPG + i]));
            }
        }

        // ---- last CTA of this unit merges the slots and leaves the transform domain
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(&a.cnt[u], 1u) == (unsigned)(c_last - c_first);
        __syncthreads();
        if (s_last) {
            __threadfence();
            const int nslots = c_last - c_first + 1;
            const float *Pu = a.part + (size_t)u * a.PMAX * HPG * PROW;
            // per-head maximum and weighted sum over the slots
            {
                const int i = tid % HPG;
                float M = -INFINITY;
                for (int sp = tid / HPG; sp < nslots; sp += NTH / HPG)
                    M = fmaxf(M, __ldcg(Pu + ((size_t)sp * HPG + i) * PROW));
                red[tid] = M;
            }
            __syncthreads();
            if (tid < HPG) {
                float M = -INFINITY;
                for (int k = tid; k < NTH; k += HPG) M = fmaxf(M, red[k]);
                cm[tid] = M;
            }
            __syncthreads();
            {
                const int i = tid % HPG;
                const float M = cm[i];
                float Ls = 0.f;
                for (int sp = tid / HPG; sp < nslots; sp += NTH / HPG) {
                    const float *Ps = Pu + ((size_t)sp * HPG + i) * PROW;
                    const float ms = __ldcg(Ps);
                    if (ms != -INFINITY) Ls = fmaf(__ldcg(Ps + 1), exp2f(ms - M), Ls);
                }
                red[tid] = Ls;
            }
            __syncthreads();
            if (tid < HPG) {
                float Ls = 0.f;
                for (int k = tid; k < NTH; k += HPG) Ls += red[k];
                cl[tid] = Ls;
            }
            __syncthreads();
            // Uv^T of this head into shared memory (one bulk copy, usually from L2)
            float *UT = reinterpret_cast<float *>(stage_base);       // [D][D]
            float *cacc = UT + D * D;                                // [HPG][D]
            float *cbar = cacc + 8 * D;                              // [HPG][D]
            if (tid == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive_expect(&ubar, D * D * 4);
                bulk_g2s(UT, a.UvT + (size_t)h * D * D, D * D * 4, &ubar);
            }
            // channel sums: thread (i, j4) sums float4 channel block j4 of head i over
            // a share of the slots; shares are added in shared memory
            for (int e = tid; e < HPG * D; e += NTH) cacc[e] = 0.f;
            __syncthreads();
            {
                const int outs = HPG * (D / 4);           // float4 outputs
                const int reps = NTH / outs > 0 ? NTH / outs : 1;
                const int o = tid % outs, rep = tid / outs;
                if (rep < reps) {
                    const int i = o / (D / 4), j4 = o % (D / 4);
                    const float M = cm[i];
                    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int sp = rep; sp < nslots; sp += reps) {
                        const float *Ps = Pu + ((size_t)sp * HPG + i) * PROW;
                        const float ms = __ldcg(Ps);
                        const float f = ms == -INFINITY ? 0.f : exp2f(ms - M);
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(Ps + 4) + j4);
                        s4.x = fmaf(v.x, f, s4.x);
                        s4.y = fmaf(v.y, f, s4.y);
                        s4.z = fmaf(v.z, f, s4.z);
                        s4.w = fmaf(v.w, f, s4.w);
                    }
                    float *dst = cacc + i * D + 4 * j4;
                    atomicAdd(dst + 0, s4.x);
                    atomicAdd(dst + 1, s4.y);
                    atomicAdd(dst + 2, s4.z);
                    atomicAdd(dst + 3, s4.w);
                }
            }
            __syncthreads();
            // the channel sums are centred: sum_i p_i (u_ij - mid_j)
            const CodecTables &tv = a.tab[h * 2 + 1];
            for (int e = tid; e < HPG * D; e += NTH) {
                const int i = e / D, j = e % D;
                const float Ls = cl[i];
                cbar[e] = (Ls > 0.f && tv.bits[j]) ? tv.step[j] * (cacc[e] / Ls) : 0.f;
            }
            const bool have_u = mbar_wait(&ubar, (uint32_t)(n_final & 1));
            ++n_final;
            if (!have_u && tid == 0) atomicOr(a.status, AATC_DEV_TIMEOUT);
            __syncthreads();
            // o = Uv cbar + mu_v
            const int Hq = a.Hkv * a.G;
            for (int e = tid; e < HPG * D; e += NTH) {
                const int i = e / D, j = e % D;
                const int gi = hg * HPG + i;
                if (gi >= a.G) continue;
                float o = 0.f;
                if (cl[i] > 0.f && have_u) {
                    const float *cb = cbar + i * D;
#pragma unroll 8
                    for (int k = 0; k < D; ++k) o = fmaf(UT[k * D + j], cb[k], o);
                    o += a.muv[h * D + j];
                }
                a.out[((size_t)b * Hq + h * a.G + gi) * D + j] = o;
            }
            if (tid == 0) a.cnt[u] = 0u;
        }
        __syncthreads();   // shared memory (tables, merge area) is reused by the next segment
    }
}

template <int GMAX, int NT, int FW>
int occupancy_of(size_t smem)
{
    auto kern = k_decode_fast<GMAX, NT, FW>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, FW * 32, smem) != cudaSuccess || n < 1) n = 1;
    return n;
}

int fast_ctas_per_sm(int groups, int NT, int FW, size_t smem)
{
    (void)FW;
    if (NT == 1) {
        if (groups <= 2) return occupancy_of<2, 1, 12>(smem);
        if (groups <= 3) return occupancy_of<3, 1, 12>(smem);
        return occupancy_of<4, 1, 12>(smem);
    }
    if (groups <= 2) return occupancy_of<2, 2, 8>(smem);
    if (groups <= 3) return occupancy_of<3, 2, 8>(smem);
    return occupancy_of<4, 2, 8>(smem);
}

// ============================================================ general path
constexpr int DEC_TILE = 128;   // tokens per tile, one thread per token
constexpr int DEC_TARGET_BLOCKS = 2 * 148;
constexpr int GEN_MAX_W = 32;

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
__global__ void k_query_prep(const T *q, int Hq, int G, const float *__restrict__ AkT,
                             const CodecTables *__restrict__ tabs, float *__restrict__ qp)
{
    __shared__ float qs[D];
    const int b = blockIdx.x, hq = blockIdx.y, j = threadIdx.x;
    const int h = hq / G;
    qs[j] = to_f32(q[((size_t)b * Hq + hq) * D + j]);
    __syncthreads();
    const float *A = AkT + (size_t)h * D * D + j;
    float acc = 0.f;
    for (int k = 0; k < D; ++k) acc = fmaf(A[(size_t)k * D], qs[k], acc);
    const CodecTables &tb = tabs[h * 2 + 0];
    qp[((size_t)b * Hq + hq) * D + j] = tb.bits[j] ? acc * tb.step[j] * 0.08838834764831845f : 0.f;
}

__device__ __forceinline__ int key_word_pos(int i, int w, int W)
{
    const int r = w >> 2, nr = min(4, W - 4 * r), ii = i & 15;
    return 16 * W * (i >> 4) + 64 * r + (ii >> 1) * 2 * nr + 2 * (w - 4 * r) + (ii & 1);
}

__device__ __forceinline__ uint32_t code_at(const uint32_t *rec, int off, int b)
{
    const int w = off >> 5, sh = off & 31;
    uint32_t v = rec[w] >> sh;
    if (sh + b > 32) v |= rec[w + 1] << (32 - sh);
    return v & ((1u << b) - 1u);
}

// One block per (split, KV head, batch row): online softmax over the block's
// token range for the G query heads of the KV head.  Partials per query head:
// m (running max of scores), l (sum of exp), acc[j] = sum_i p_i u^V_ij.
__global__ void __launch_bounds__(DEC_TILE) k_decode_split_general(
    const float *__restrict__ qp, const uint32_t *__restrict__ kp, const uint32_t *__restrict__ vp,
    int L_cap, const int32_t *__restrict__ seq_lens, int L, int Hkv, int G, int W, int chunk,
    int n_split, const HeadPlan *__restrict__ plans, const CodecTables *__restrict__ tabs,
    float *__restrict__ part)
{
    __shared__ float q_s[AATC_MAX_G][D];
    __shared__ float p_s[DEC_TILE][AATC_MAX_G + 1];
    __shared__ uint8_t v_s[DEC_TILE][D + 4];
    __shared__ int16_t offk[D], offv[D];
    __shared__ uint8_t bk[D], bv[D];
    __shared__ float red[4][AATC_MAX_G];
    __shared__ float m_s[AATC_MAX_G], alpha_s[AATC_MAX_G];

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    const int len = seq_lens ? min(max(seq_lens[b], 0), L) : L;
    const int begin = split * chunk, end = min(begin + chunk, len);
    const int Hq = Hkv * G;
    for (int e = t; e < G * D; e += DEC_TILE) {
        int gg = e / D, j = e % D;
        q_s[gg][j] = qp[((size_t)b * Hq + h * G + gg) * D + j];
    }
    {
        const HeadPlan &pk = plans[h * 2 + 0], &pv = plans[h * 2 + 1];
        offk[t] = pk.off[t];
        offv[t] = pv.off[t];
    }
    __syncthreads();
    bk[t] = tabs[h * 2 + 0].bits[t];
    bv[t] = tabs[h * 2 + 1].bits[t];
    if (t < AATC_MAX_G) m_s[t] = -INFINITY;
    __syncthreads();

    float acc[AATC_MAX_G], lsum[AATC_MAX_G];
#pragma unroll
    for (int gg = 0; gg < AATC_MAX_G; ++gg) { acc[gg] = 0.f; lsum[gg] = 0.f; }

    const size_t base = ((size_t)b * Hkv + h) * (size_t)L_cap * W;
    for (int tok0 = begin; tok0 < end; tok0 += DEC_TILE) {
        const int tok = tok0 + t;
        const bool valid = tok < end;
        uint32_t rec[GEN_MAX_W + 1];
        float sc[AATC_MAX_G];
#pragma unroll
        for (int gg = 0; gg < AATC_MAX_G; ++gg) sc[gg] = -INFINITY;
        if (valid) {
            const uint32_t *tile = kp + base + (size_t)(tok >> 5) * 32 * W;
            for (int w = 0; w < W; ++w) rec[w] = tile[key_word_pos(tok & 31, w, W)];
            rec[W] = 0u;
#pragma unroll
            for (int gg = 0; gg < AATC_MAX_G; ++gg) sc[gg] = 0.f;
            for (int j = 0; j < D; ++j) {
                if (!bk[j]) continue;
                const float u = (float)code_at(rec, offk[j], bk[j]);
#pragma unroll
                for (int gg = 0; gg < AATC_MAX_G; ++gg)
                    if (gg < G) sc[gg] = fmaf(q_s[gg][j], u, sc[gg]);
            }
            const uint32_t *vt = vp + base + (size_t)(tok >> 5) * 32 * W;
            for (int w = 0; w < W; ++w) {
                const uint32_t lo = (vt[16 * (2 * w) + ((tok & 31) >> 1)] >> (16 * (tok & 1))) & 0xFFFFu;
                const uint32_t hi = (vt[16 * (2 * w + 1) + ((tok & 31) >> 1)] >> (16 * (tok & 1))) & 0xFFFFu;
                rec[w] = lo | (hi << 16);
            }
            rec[W] = 0u;
            for (int j = 0; j < D; ++j) v_s[t][j] = bv[j] ? (uint8_t)code_at(rec, offv[j], bv[j]) : 0;
        } else {
            for (int j = 0; j < D; ++j) v_s[t][j] = 0;
        }
#pragma unroll
        for (int gg = 0; gg < AATC_MAX_G; ++gg) {
            float mx = sc[gg];
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) red[warp][gg] = mx;
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
        for (int gg = 0; gg < AATC_MAX_G; ++gg)
            if (gg < G) p_s[t][gg] = (valid && m_s[gg] != -INFINITY) ? __expf(sc[gg] - m_s[gg]) : 0.f;
        __syncthreads();
#pragma unroll
        for (int gg = 0; gg < AATC_MAX_G; ++gg)
            if (gg < G) { acc[gg] *= alpha_s[gg]; lsum[gg] *= alpha_s[gg]; }
        for (int i = 0; i < DEC_TILE; ++i) {
            const float u = (float)v_s[i][t];
#pragma unroll
            for (int gg = 0; gg < AATC_MAX_G; ++gg)
                if (gg < G) { acc[gg] = fmaf(p_s[i][gg], u, acc[gg]); lsum[gg] += p_s[i][gg]; }
        }
        __syncthreads();
    }
#pragma unroll
    for (int gg = 0; gg < AATC_MAX_G; ++gg) {
        if (gg >= G) break;
        float *P = part + (((size_t)b * Hq + h * G + gg) * n_split + split) * (2 + D);
        P[2 + t] = acc[gg];
        if (t == 0) { P[0] = m_s[gg]; P[1] = lsum[gg]; }
    }
}

// One block per (batch row, query head): LSE-merge the splits (natural-log
// maxima), leave the transform domain, apply Uv and add mu_v.  A row with no
// tokens gets zeros.
__global__ void k_decode_combine(const float *__restrict__ part, int n_split, int Hq, int G,
                                 const CodecTables *__restrict__ tabs, const float *__restrict__ UvT,
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
        const float *U = UvT + (size_t)h * D * D + j;
        for (int k = 0; k < D; ++k) o = fmaf(U[(size_t)k * D], cbar[k], o);
        o += muv[h * D + j];
    }
    out[((size_t)b * Hq + hq) * D + j] = o;
}

size_t general_ws_bytes(const aatc_calib *h, int B, int L)
{
    SplitPlan p = plan_splits(B, h->Hkv, L);
    size_t qp = (size_t)B * h->Hq * D * sizeof(float);
    size_t part = (size_t)B * h->Hq * p.n_split * (2 + D) * sizeof(float);
    return ((qp + 255) / 256) * 256 + part;
}

template <int GMAX, int NT, int FW>
aatc_status launch_fast(const FastGeom &f, const FastArgs &a, cudaStream_t s)
{
    auto kern = k_decode_fast<GMAX, NT, FW>;
    AATC_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f.smem));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(f.C);
    cfg.blockDim = dim3(FW * 32);
    cfg.dynamicSmemBytes = f.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    AATC_CUDA(cudaLaunchKernelEx(&cfg, kern, a));
    return AATC_OK;
}

}  // namespace

size_t decode_ws_bytes(const aatc_calib *h, int B, int L)
{
    if (fast_ok(h)) return fast_geom(h, B, L).ws_total;
    return general_ws_bytes(h, B, L);
}

aatc_status decode_run(const aatc_calib *h, const void *q, const uint32_t *kp, const uint32_t *vp,
                       int L_cap, const int32_t *seq_lens, int L, int B, float *out, void *ws,
                       size_t ws_bytes, cudaStream_t s)
{
    if (B == 0) return AATC_OK;
    (void)ws_bytes;
    if (fast_ok(h)) {
        const FastGeom f = fast_geom(h, B, L);
        if ((long)B * f.HG > 65535)
            return aatc_fail(AATC_ERR_UNSUPPORTED, "batch %d too large for GQA group %d", B, h->G);
        if (f.n_tiles == 0) {   // nothing to attend: zeros
            AATC_CUDA(cudaMemsetAsync(out, 0, (size_t)B * h->Hq * D * sizeof(float), s));
            return AATC_OK;
        }
        char *w = (char *)ws;
        uint32_t *qtab = (uint32_t *)w;
        float *qsc = (float *)(w + f.ws_qtab);
        float *part = (float *)(w + f.ws_qtab + f.ws_qsc);
        uint32_t *cnt = (uint32_t *)(w + f.ws_qtab + f.ws_qsc + f.ws_part);
        const dim3 pg(B, h->Hkv, f.HG);
        if (h->dtype == AATC_BF16)
        {
            auto kq = k_qprep_fast<__nv_bfloat16>;
            AATC_CUDA(cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QP_SMEM));
            kq<<<pg, QP_THREADS, QP_SMEM, s>>>((const __nv_bfloat16 *)q, h->AkT32, h->UvT32, h->tab, h->plan,
                                               h->Hkv, h->G, f.HG, f.HPG, f.NT, f.ksteps, qtab, qsc, cnt,
                                               h->status);
        }
        else {
            auto kq = k_qprep_fast<float>;
            AATC_CUDA(cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QP_SMEM));
            kq<<<pg, QP_THREADS, QP_SMEM, s>>>((const float *)q, h->AkT32, h->UvT32, h->tab, h->plan, h->Hkv,
                                               h->G, f.HG, f.HPG, f.NT, f.ksteps, qtab, qsc, cnt, h->status);
        }
        AATC_CUDA(cudaGetLastError());
        FastArgs a;
        a.kp = kp;
        a.vp = vp;
        a.seq_lens = seq_lens;
        a.L = L;
        a.L_cap = L_cap;
        a.W = h->W;
        a.rows = f.rows;
        a.groups = f.groups;
        a.Hkv = h->Hkv;
        a.G = h->G;
        a.HG = f.HG;
        a.HPG = f.HPG;
        a.n_tiles = f.n_tiles;
        a.units = f.units;
        a.C = f.C;
        a.PMAX = f.PMAX;
        a.plan = h->plan;
        a.qtab = qtab;
        a.qsc = qsc;
        a.part = part;
        a.cnt = cnt;
        a.tab = h->tab;
        a.UvT = h->UvT32;
        a.muv = h->muv32;
        a.out = out;
        a.status = h->status;
        if (f.NT == 1) {
            if (f.groups <= 2) return launch_fast<2, 1, 12>(f, a, s);
            if (f.groups <= 3) return launch_fast<3, 1, 12>(f, a, s);
            return launch_fast<4, 1, 12>(f, a, s);
        }
        if (f.groups <= 2) return launch_fast<2, 2, 8>(f, a, s);
        if (f.groups <= 3) return launch_fast<3, 2, 8>(f, a, s);
        return launch_fast<4, 2, 8>(f, a, s);
    }
    if (h->W > GEN_MAX_W) return aatc_fail(AATC_ERR_UNSUPPORTED, "record of %d words", h->W);
    SplitPlan p = plan_splits(B, h->Hkv, L);
    float *qp = (float *)ws;
    size_t qp_bytes = (((size_t)B * h->Hq * D * sizeof(float) + 255) / 256) * 256;
    float *part = (float *)((char *)ws + qp_bytes);
    if (h->dtype == AATC_BF16)
        k_query_prep<__nv_bfloat16><<<dim3(B, h->Hq), D, 0, s>>>((const __nv_bfloat16 *)q, h->Hq, h->G,
                                                                 h->AkT32, h->tab, qp);
    else
        k_query_prep<float><<<dim3(B, h->Hq), D, 0, s>>>((const float *)q, h->Hq, h->G, h->AkT32, h->tab, qp);
    k_decode_split_general<<<dim3(p.n_split, h->Hkv, B), DEC_TILE, 0, s>>>(
        qp, kp, vp, L_cap, seq_lens, L, h->Hkv, h->G, h->W, p.chunk, p.n_split, h->plan, h->tab, part);
    k_decode_combine<<<dim3(B, h->Hq), D, 0, s>>>(part, p.n_split, h->Hq, h->G, h->tab, h->UvT32,
                                                  h->muv32, out);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

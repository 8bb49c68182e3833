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
//   k_decode_fast   one persistent CTA per SM over a balanced share of all
//                   (batch row, KV head, head group, 32-token tile) work.  Per
//                   segment it computes q' for the head group and expands it
//                   to one fp16 hi/lo weight per record piece in mma.sync
//                   B-fragment order; each warp streams its own tiles into
//                   shared memory with cp.async.bulk, unpacks pieces with one
//                   AND per two fp16 operands, runs scores and P.V on mma.sync
//                   (fp16 hi/lo operands, fp32 accumulation) with an exp2
//                   online softmax; warps merge by log-sum-exp into one
//                   partial per segment.
//   k_decode_combine_fast  per (batch row, KV head, head group), launched
//                   with programmatic dependent launch: merges the partials
//                   and applies Uv once per head.
// General path (any shape): one thread per token, codes read by offset.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <mutex>

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

// Work split: every (batch row, KV head, head group) is a "unit" of
// n_tiles = ceil(L/32) tiles, cut into S = max(1, resident CTAs / units)
// equal contiguous ranges; CTA (unit u, split s) streams range s of unit u
// and leaves partial slot s.
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
    int S;           // splits (CTAs, partial slots) per unit
    int tiles_per;   // tiles per split
    size_t stage_bytes, smem, ws_part, ws_total;
};

size_t fast_smem(int FW, int W, int groups, int HPG, int NT, int ksteps, int rows)
{
    const size_t SB = 256 * (size_t)W + 512;
    const size_t rows_tot = 64 * (size_t)groups;
    const size_t merge = (size_t)FW * (rows_tot + 2) * HPG * 4 + (size_t)D * HPG * 4;
    size_t big = (size_t)FW * FSTAGES * SB;
    big = big > merge ? big : merge;
    big = (big + 127) & ~(size_t)127;
    return big + (size_t)FW * FSTAGES * 8 + (size_t)FW * 16 * PSTRIDE * 2 + (size_t)ksteps * NT * 32 * 8 +
           (size_t)rows * 4 * 8 * 4 + (size_t)groups * 64 * 4 + 256 * 2 + 8 * 4 + 2 * 8 * D * 4 + 256 * 2 + 16;
}

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
    const int C = sm_count() * per_sm;
    f.S = C / f.units > 1 ? C / f.units : 1;
    if (f.S > f.n_tiles) f.S = f.n_tiles > 0 ? f.n_tiles : 1;
    f.tiles_per = f.n_tiles > 0 ? (f.n_tiles + f.S - 1) / f.S : 1;
    f.S = f.n_tiles > 0 ? (f.n_tiles + f.tiles_per - 1) / f.tiles_per : 1;
    f.stage_bytes = 256 * (size_t)h->W + 512;
    f.ws_part = (((size_t)f.units * f.S * f.HPG * PROW * 4) + 255) & ~(size_t)255;
    f.ws_total = f.ws_part;
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
    // each try may suspend the thread for up to ~20 us until the phase completes
    for (int it = 0; it < (1 << 16); ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(parity), "r"(20000)
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
    int L, L_cap, W, rows, groups, Hkv, G, HG, HPG, n_tiles, units, S, tiles_per;
    const HeadPlan *plan;
    const void *q;          // [B][Hq][D] of the handle's dtype
    const float *AkT;       // [Hkv][D][D]
    float *part;            // [units][S][HPG][PROW]
    const CodecTables *tab;
    uint32_t *status;
};

template <int GMAX, int NT, int FW, typename QT>
__global__ void __launch_bounds__(FW * 32) k_decode_fast(FastArgs a)
{
    constexpr int NTH = FW * 32;
    asm volatile("griddepcontrol.launch_dependents;");   // the combine kernel may start its prologue
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
    big = (big + 127) & ~(size_t)127;
    unsigned char *stage_base = smem;
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + big);
    __half *pbuf = reinterpret_cast<__half *>(mbar + FW * FSTAGES);
    uint2 *qtab_s = reinterpret_cast<uint2 *>(pbuf + FW * 16 * PSTRIDE);
    uint32_t *kmask_s = reinterpret_cast<uint32_t *>(qtab_s + ksteps * NT * 32);
    uint32_t *vmask_s = kmask_s + rows * 4 * 8;
    int16_t *vrow_s = reinterpret_cast<int16_t *>(vmask_s + groups * 64);   // [groups*64] (ch << 8 | ex + 64)
    float *sc_s = reinterpret_cast<float *>(vrow_s + 256);
    float *qs = sc_s + 8;                     // [8][D] query rows of the head group
    float *pa = qs + 8 * D;                   // [8][D] q' of the head group
    int16_t *slot_s = reinterpret_cast<int16_t *>(pa + 8 * D);   // [16][8][2] key piece: ch | (ex + 64) << 8
    __shared__ float cm[8], cl[8], cs[8][FW];
    __shared__ float S_s[8];
    __shared__ float ksc_s[D];                 // Delta_K / sqrt(d), 0 for pruned channels
    __shared__ float vmid_s[256];              // value piece midpoints (2^w-1)/2 * 2^(p-24), per row

    uint64_t *my_mbar = mbar + warp * FSTAGES;
    unsigned char *my_stage = stage_base + (size_t)warp * FSTAGES * SB;
    const uint32_t tile_bytes = 128u * W;
    if (lane == 0) {
        for (int s = 0; s < FSTAGES; ++s) mbar_init(&my_mbar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // The warp's n-th tile (over all its segments) goes through stage n % FSTAGES
    // and completes phase n / FSTAGES of that stage's barrier.
    int n_issued = 0, n_done = 0;

    {
        // ---- this CTA: unit u, split sp, tiles [ta, tb) of the unit
        const int u = blockIdx.x / a.S, sp = blockIdx.x % a.S;
        const int ta = sp * a.tiles_per, tb = min(ta + a.tiles_per, a.n_tiles);
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

        // ---- tables of this unit and its query weights.  All global loads of
        // the prologue are issued before any is used: one round trip.
        const HeadPlan &pk = a.plan[h * 2 + 0];
        const HeadPlan &pv = a.plan[h * 2 + 1];
        {
            // A_k^T: thread (k-set kq, channel quad j4) holds rows k = kq + NTH/32 * m
            constexpr int KSTEP = NTH / 32;
            constexpr int KPER = (D + KSTEP - 1) / KSTEP;
            const int j4 = tid & 31, kq = tid >> 5;
            float4 av[KPER];
            const float4 *Ag = reinterpret_cast<const float4 *>(a.AkT + (size_t)h * D * D) + j4;
#pragma unroll
            for (int m = 0; m < KPER; ++m) {
                const int k = kq + KSTEP * m;
                av[m] = k < D ? __ldg(Ag + (size_t)k * (D / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            const QT *qg = reinterpret_cast<const QT *>(a.q);
            const int Hq = a.Hkv * a.G;
            // every global load of the prologue is issued before any result is stored
            constexpr int QPER = (8 * D + NTH - 1) / NTH;
            float qv[QPER];
#pragma unroll
            for (int r = 0; r < QPER; ++r) {
                const int e = tid + r * NTH;
                const int i = e >> 7, cc = e & (D - 1), gi = hg * HPG + i;
                qv[r] = (e < 8 * D && i < HPG && gi < a.G) ? to_f32(qg[((size_t)b * Hq + h * a.G + gi) * D + cc]) : 0.f;
            }
            const int ek = tid;                       // rows * 32 <= NTH
            const uint32_t km = ek < rows * 32 ? pk.mask[ek >> 3][ek & 7] : 0u;
            constexpr int VPER = (4 * 64 + NTH - 1) / NTH;
            uint32_t vm[VPER];
            int vch[VPER], vex[VPER];
#pragma unroll
            for (int r = 0; r < VPER; ++r) {
                const int e = tid + r * NTH;
                const int gr = e >> 6, m4 = (e >> 4) & 3, rr = e & 15;
                const int hw = 8 * gr + (rr & 7), k = 2 * m4 + (rr >> 3);
                const bool in = e < groups * 64;
                vm[r] = in ? pv.mask[e >> 3][e & 7] : 0u;
                vch[r] = in ? pv.ch[hw][k][0] : -1;
                vex[r] = in ? pv.ex[hw][k][0] : 0;
            }
            const int es = tid;                       // 16 * 16 <= NTH
            int sch = -1, sex = 0;
            if (es < 256) {
                sch = pk.ch[es >> 4][(es >> 1) & 7][es & 1];
                sex = pk.ex[es >> 4][(es >> 1) & 7][es & 1];
            }
            const CodecTables &tk = a.tab[h * 2 + 0];
            const float ksc = tid < D ? (tk.bits[tid] ? tk.step[tid] * 0.08838834764831845f : 0.f) : 0.f;
            // ... then stored
#pragma unroll
            for (int r = 0; r < QPER; ++r) {
                const int e = tid + r * NTH;
                if (e < 8 * D) {
                    qs[e] = qv[r];
                    pa[e] = 0.f;
                }
            }
            if (ek < rows * 32) kmask_s[ek] = km;
#pragma unroll
            for (int r = 0; r < VPER; ++r) {
                const int e = tid + r * NTH;
                if (e < groups * 64) {
                    vmask_s[e] = vm[r];
                    // row e = (group, m4, rr): half-word 8 group + rr%8, slot 2 m4 + rr/8; the
                    // slot's mask holds (2^w - 1) << p per half: low half / 2 = midpoint * 2^p
                    const int gr = e >> 6, m4 = (e >> 4) & 3, rr = e & 15;
                    const int hw = 8 * gr + (rr & 7), k = 2 * m4 + (rr >> 3);
                    (void)hw;
                    (void)k;
                    vrow_s[e] = (int16_t)(vch[r] < 0 ? -1 : (vch[r] << 8) | (vex[r] + 64));
                    vmid_s[e] = 0.f;
                }
            }
            if (es < 256) slot_s[es] = (int16_t)(sch < 0 ? -1 : (sch | ((sex + 64) << 8)));
            if (tid < D) ksc_s[tid] = ksc;
            __syncthreads();
            for (int e = tid; e < groups * 64; e += NTH) {
                const int gr = e >> 6, m4 = (e >> 4) & 3, rr = e & 15;
                const int hw = 8 * gr + (rr & 7), k = 2 * m4 + (rr >> 3);
                vmid_s[e] = ldexpf((float)(vmask_s[hw * 8 + k] & 0xFFFFu), -25);
            }
            // q'_i[j] = sum_k A_k[j][k] q_i[k]: partial sums over this thread's rows
            float4 acc4[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < KPER; ++m) {
                const int k = kq + KSTEP * m;
                if (k >= D) break;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i >= HPG) break;
                    const float qv = qs[i * D + k];
                    acc4[i].x = fmaf(av[m].x, qv, acc4[i].x);
                    acc4[i].y = fmaf(av[m].y, qv, acc4[i].y);
                    acc4[i].z = fmaf(av[m].z, qv, acc4[i].z);
                    acc4[i].w = fmaf(av[m].w, qv, acc4[i].w);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i >= HPG) break;
                float *d = pa + i * D + 4 * j4;
                atomicAdd(d + 0, acc4[i].x);
                atomicAdd(d + 1, acc4[i].y);
                atomicAdd(d + 2, acc4[i].z);
                atomicAdd(d + 3, acc4[i].w);
            }
            __syncthreads();
            for (int e = tid; e < HPG * D; e += NTH) pa[e] *= ksc_s[e & (D - 1)];
            __syncthreads();
            if (warp < HPG) {   // warp i: largest |q'| of head i -> power-of-two scale
                float mx = 0.f;
                for (int k = lane; k < D; k += 32) mx = fmaxf(mx, fabsf(pa[warp * D + k]));
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (lane == 0) {
                    // pieces carry 2^ex with ex <= 7: keep mx * 2^7 * S below 2^13
                    int e = 0;
                    if (mx > 0.f) frexpf(mx, &e);
                    const float S = mx > 0.f ? ldexpf(1.f, 6 - e) : 1.f;
                    S_s[warp] = S;
                    sc_s[warp] = ldexpf(1.f, 24) / S * LOG2E;
                }
            }
            __syncthreads();
            // B fragments: entry (kstep, n-tile t, lane) = (b0, b1), column n = 8t + lane/4 =
            // (head n/2, hi if n even else lo), k-step (r, s) from record word 4r + lane%4,
            // slots 2s (b0) and 2s+1 (b1), low half first; weight = q'_ch * 2^ex * S
            for (int en = tid; en < ksteps * NT * 32; en += NTH) {
                const int ln = en & 31, t = (en >> 5) % NT, ks = (en >> 5) / NT;
                const int r = ks >> 2, s4 = ks & 3;
                const int n = 8 * t + (ln >> 2), i = n >> 1, part = n & 1;
                const int w = 4 * r + (ln & 3);
                uint32_t o2[2];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int k = 2 * s4 + rr;
                    float v2[2];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int sl = slot_s[(w * 8 + k) * 2 + half];
                        float val = 0.f;
                        if (sl >= 0 && i < HPG && hg * HPG + i < a.G)
                            val = ldexpf(pa[i * D + (sl & 255)] * S_s[i], (sl >> 8) - 64);
                        const float hi = __half2float(__float2half_rn(val));
                        v2[half] = part ? val - hi : hi;
                    }
                    o2[rr] = pack_half2(v2[0], v2[1]);
                }
                qtab_s[en] = make_uint2(o2[0], o2[1]);
            }
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

            // ---- scores: rows = tokens (row g: 2g, row g+8: 2g+1 of the half), k = record pieces;
            // one accumulator chain per (half, record row) for independent MMAs
            float C[2][NT][4];
            {
                float Cr[2][4][NT][4];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int t = 0; t < NT; ++t)
#pragma unroll
                            for (int k = 0; k < 4; ++k) Cr[hf][r][t][k] = 0.f;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (r >= rows) break;
                    const int nr = min(4, W - 4 * r);
                    const uint4 mA = *reinterpret_cast<const uint4 *>(kmask_s + (4 * r + c) * 8);
                    const uint4 mB = *reinterpret_cast<const uint4 *>(kmask_s + (4 * r + c) * 8 + 4);
                    const uint32_t mk[8] = {mA.x, mA.y, mA.z, mA.w, mB.x, mB.y, mB.z, mB.w};
                    uint32_t x0[2], x1[2], y0[2], y1[2];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const uint2 kw =
                            *reinterpret_cast<const uint2 *>(Kt + hf * 16 * W + 64 * r + g * 2 * nr + 2 * c);
                        x0[hf] = kw.x;
                        x1[hf] = kw.y;
                        y0[hf] = kw.x >> 8;
                        y1[hf] = kw.y >> 8;
                    }
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        uint2 bq[NT];
#pragma unroll
                        for (int t = 0; t < NT; ++t) bq[t] = qtab_s[((r * 4 + s4) * NT + t) * 32 + lane];
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const uint32_t sa = s4 < 2 ? x0[hf] : y0[hf], sb = s4 < 2 ? x1[hf] : y1[hf];
                            const uint32_t A0 = sa & mk[2 * s4], A1 = sb & mk[2 * s4];
                            const uint32_t A2 = sa & mk[2 * s4 + 1], A3 = sb & mk[2 * s4 + 1];
#pragma unroll
                            for (int t = 0; t < NT; ++t) mma16816(Cr[hf][r][t], A0, A1, A2, A3, bq[t].x, bq[t].y);
                        }
                    }
                }
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int t = 0; t < NT; ++t)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            C[hf][t][k] = (Cr[hf][0][t][k] + Cr[hf][1][t][k]) + (Cr[hf][2][t][k] + Cr[hf][3][t][k]);
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
        {
            float *P = a.part + ((size_t)u * a.S + sp) * HPG * PROW;
            for (int e = tid; e < HPG * PROW; e += NTH) {
                const int i = e / PROW, j = e % PROW;
                P[e] = j == 0 ? cm[i] : (j == 1 ? cl[i] : (j < 4 ? 0.f : ach[(j - 4) * HPG + i]));
            }
        }
    }
}


// Merge the slots of one unit and leave the transform domain:
//   o = Uv (Delta_V o sum_i p_i (u_i - mid) / sum_i p_i) + mu_v
// (the slots hold centred sums).  Launched after k_decode_fast with
// programmatic dependent launch: Uv^T and the tables are staged before the
// wait for the split kernel's partials.
constexpr int CB_THREADS = 256;
constexpr size_t CB_SMEM = (size_t)D * D * 4;
__global__ void __launch_bounds__(CB_THREADS) k_decode_combine_fast(
    const float *__restrict__ part, int S, int Hkv, int G, int HG, int HPG,
    const CodecTables *__restrict__ tabs, const float *__restrict__ UvT, const float *__restrict__ muv,
    float *__restrict__ out)
{
    extern __shared__ __align__(16) float UT[];          // [D][D]
    __shared__ float cacc[8][D], cbar[8][D];
    __shared__ float sM[8], sL[8];
    __shared__ float step_s[D], muv_s[D];
    __shared__ float ml_s[2][CB_THREADS];
    const int u = blockIdx.x, tid = threadIdx.x;
    const int b = u / (Hkv * HG), h = (u / HG) % Hkv, hg = u % HG;
    {
        // every load of the prologue in flight at once
        const float4 *src = reinterpret_cast<const float4 *>(UvT + (size_t)h * D * D);
        float4 ut[D * D / 4 / CB_THREADS];
#pragma unroll
        for (int r = 0; r < D * D / 4 / CB_THREADS; ++r) ut[r] = __ldg(src + tid + r * CB_THREADS);
        const CodecTables &tv = tabs[h * 2 + 1];
        float st = 0.f, mv = 0.f;
        if (tid < D) {
            st = tv.bits[tid] ? tv.step[tid] : 0.f;
            mv = muv[h * D + tid];
        }
        float4 *dst = reinterpret_cast<float4 *>(UT);
#pragma unroll
        for (int r = 0; r < D * D / 4 / CB_THREADS; ++r) dst[tid + r * CB_THREADS] = ut[r];
        if (tid < D) {
            step_s[tid] = st;
            muv_s[tid] = mv;
        }
        for (int e = tid; e < 8 * D; e += CB_THREADS) (&cacc[0][0])[e] = 0.f;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");   // partials of k_decode_fast
    const int nslots = S;
    const float *Pu = part + (size_t)u * S * HPG * PROW;
    // per-head maximum and weighted sum over the slots; (slot, head) pairs in parallel
    float Mh = -INFINITY;
    for (int e0 = 0; e0 < nslots * HPG; e0 += CB_THREADS) {
        const int e = e0 + tid;
        float m = -INFINITY, l = 0.f;
        if (e < nslots * HPG) {
            m = __ldcg(Pu + (size_t)e * PROW);
            l = __ldcg(Pu + (size_t)e * PROW + 1);
        }
        __syncthreads();
        ml_s[0][tid] = m;
        ml_s[1][tid] = l;
        __syncthreads();
        if (tid < HPG) {
            const int cnt = min(CB_THREADS, nslots * HPG - e0);
            float M = Mh, Ls = e0 == 0 ? 0.f : sL[tid];
            for (int k = tid; k < cnt; k += HPG) {
                const float mk = ml_s[0][k];
                if (mk == -INFINITY) continue;
                if (mk > M) {
                    Ls = (M == -INFINITY) ? 0.f : Ls * exp2f(M - mk);
                    M = mk;
                }
                Ls = fmaf(ml_s[1][k], exp2f(mk - M), Ls);
            }
            Mh = M;
            sM[tid] = M;
            sL[tid] = Ls;
        }
    }
    __syncthreads();
    {   // thread (rep, i, j4): float4 block j4 of head i over every reps-th slot
        const int outs = HPG * (D / 4);
        const int reps = CB_THREADS / outs;
        const int o = tid % outs, rep = tid / outs;
        const int i = o / (D / 4), j4 = o % (D / 4);
        const float M = sM[i];
        float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
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
        atomicAdd(&cacc[i][4 * j4 + 0], s4.x);
        atomicAdd(&cacc[i][4 * j4 + 1], s4.y);
        atomicAdd(&cacc[i][4 * j4 + 2], s4.z);
        atomicAdd(&cacc[i][4 * j4 + 3], s4.w);
    }
    __syncthreads();
    for (int e = tid; e < HPG * D; e += CB_THREADS) {
        const int i = e / D, j = e % D;
        cbar[i][j] = sL[i] > 0.f ? step_s[j] * (cacc[i][j] / sL[i]) : 0.f;
    }
    __syncthreads();
    const int Hq = Hkv * G;
    for (int e = tid; e < HPG * D; e += CB_THREADS) {
        const int i = e / D, j = e % D, gi = hg * HPG + i;
        if (gi >= G) continue;
        float o = 0.f;
        if (sL[i] > 0.f) {
#pragma unroll 8
            for (int k = 0; k < D; ++k) o = fmaf(UT[k * D + j], cbar[i][k], o);
            o += muv_s[j];
        }
        out[((size_t)b * Hq + h * G + gi) * D + j] = o;
    }
}

template <int GMAX, int NT, int FW>
int occupancy_of(size_t smem)
{
    auto kern = k_decode_fast<GMAX, NT, FW, __nv_bfloat16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, FW * 32, smem) != cudaSuccess || n < 1) n = 1;
    return n;
}

int fast_ctas_per_sm_uncached(int groups, int NT, size_t smem)
{
    if (NT == 1) {
        if (groups <= 2) return occupancy_of<2, 1, 12>(smem);
        if (groups <= 3) return occupancy_of<3, 1, 12>(smem);
        return occupancy_of<4, 1, 12>(smem);
    }
    if (groups <= 2) return occupancy_of<2, 2, 8>(smem);
    if (groups <= 3) return occupancy_of<3, 2, 8>(smem);
    return occupancy_of<4, 2, 8>(smem);
}

int fast_ctas_per_sm(int groups, int NT, int FW, size_t smem)
{
    // the answer depends only on the kernel variant and its shared memory
    static struct { int groups, NT, FW; size_t smem; int n; } cache[16];
    static int used = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].groups == groups && cache[i].NT == NT && cache[i].FW == FW && cache[i].smem == smem)
            return cache[i].n;
    const int n = fast_ctas_per_sm_uncached(groups, NT, smem);
    if (used < 16) cache[used++] = {groups, NT, FW, smem, n};
    return n;
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

// Raise a kernel's dynamic shared memory limit once per kernel (and per
// larger size seen).  Keyed by the kernel's address: every instance of a
// template has the same function type.
aatc_status smem_limit(const void *kern, size_t bytes)
{
    static struct { const void *k; size_t set; } seen[32];
    static int used = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int i = 0;
    while (i < used && seen[i].k != kern) ++i;
    if (i < used && seen[i].set >= bytes) return AATC_OK;
    AATC_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
    if (i == used && used < 32) seen[used++] = {kern, 0};
    if (i < used) seen[i].set = bytes;
    return AATC_OK;
}

template <int GMAX, int NT, int FW>
aatc_status launch_fast(const FastGeom &f, const FastArgs &a, aatc_dtype dt, cudaStream_t s)
{
    if (dt == AATC_BF16) {
        auto kern = k_decode_fast<GMAX, NT, FW, __nv_bfloat16>;
        aatc_status st = smem_limit((const void *)kern, f.smem);
        if (st != AATC_OK) return st;
        kern<<<f.units * f.S, FW * 32, f.smem, s>>>(a);
    } else {
        auto kern = k_decode_fast<GMAX, NT, FW, float>;
        aatc_status st = smem_limit((const void *)kern, f.smem);
        if (st != AATC_OK) return st;
        kern<<<f.units * f.S, FW * 32, f.smem, s>>>(a);
    }
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

aatc_status launch_combine(const FastGeom &f, const aatc_calib *h, const float *part, float *out, cudaStream_t s)
{
    aatc_status st0 = smem_limit((const void *)k_decode_combine_fast, CB_SMEM);
    if (st0 != AATC_OK) return st0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(f.units);
    cfg.blockDim = dim3(CB_THREADS);
    cfg.dynamicSmemBytes = CB_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    AATC_CUDA(cudaLaunchKernelEx(&cfg, k_decode_combine_fast, part, f.S, h->Hkv, h->G, f.HG, f.HPG,
                                 (const CodecTables *)h->tab, (const float *)h->UvT32, (const float *)h->muv32,
                                 out));
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
        float *part = (float *)ws;
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
        a.S = f.S;
        a.tiles_per = f.tiles_per;
        a.plan = h->plan;
        a.q = q;
        a.AkT = h->AkT32;
        a.part = part;
        a.tab = h->tab;
        a.status = h->status;
        aatc_status st;
        if (f.NT == 1) {
            if (f.groups <= 2) st = launch_fast<2, 1, 12>(f, a, h->dtype, s);
            else if (f.groups <= 3) st = launch_fast<3, 1, 12>(f, a, h->dtype, s);
            else st = launch_fast<4, 1, 12>(f, a, h->dtype, s);
        } else {
            if (f.groups <= 2) st = launch_fast<2, 2, 8>(f, a, h->dtype, s);
            else if (f.groups <= 3) st = launch_fast<3, 2, 8>(f, a, h->dtype, s);
            else st = launch_fast<4, 2, 8>(f, a, h->dtype, s);
        }
        if (st != AATC_OK) return st;
        return launch_combine(f, h, part, out, s);
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

// encode_tc.cu -- tensor-core encoder for bf16 keys/values.
//
// Transform, quantize and bit-pack ("Attention-Aware Transform Coding Guide:
// KV Compression", section "End-to-End Implementation": rotate into the
// calibrated basis, quantize each channel at its allocated width; "Spend
// Bits Where Queries Look", Abstract: fixed per-token bit count).
//
// The transform c = T x of a 128-token block is a dense 128 x 128 x 128
// contraction, done by tcgen05.mma: A = the bf16 token rows (exact), B = T
// split in three bf16 terms T1 + T2 + T3 (about 24 significant bits, so c is
// as accurate as an fp32 product), accumulated in fp32 in tensor memory.
// T's rows are stored in record order, so accumulator column n is the code
// at record position n and the epilogue packs codes front to back.
//
// One persistent CTA per SM works through a contiguous range of (head,
// tensor, batch row, 128-token block) items:
//   warp 17, one thread: TMA loads of the x tiles (ES = 3 stages where shared
//       memory allows, i.e. records of up to 12 words, else 2), each stage
//       refilled as soon as the MMAs of its previous item are done with it;
//   warp 16, one thread: TMA loads of T (once per head and tensor) and MMA
//       issue into NGRP = 4 tensor-memory accumulators, item n into
//       accumulator n % 4;
//   warps 0-15: four epilogue groups of four warps; group g takes items
//       g, g + 4, ..., thread = token = tensor-memory lane: read the 128
//       accumulators, quantize (v = c inv + off, clamp, round half to even),
//       pack LSB-first into the record and place the words in the tiled
//       cache layout in shared memory; full aligned blocks leave by one bulk
//       store, other blocks by per-token stores.
// Packing: rounding adds 1.5 * 2^23, after which the float's bit pattern is
// 0x4B400000 + code.  That pattern, times 2^(bit position), is added into the
// record word as it is (one integer multiply-add per code); the constant
// parts add up to a per-word constant fixed by the bit plan (wfix), taken off
// as the word leaves.  A code that crosses into the next word carries its
// high part over by a high multiply (the constant's high part is in the next
// word's wfix).
// Every wait is bounded; a wait that gives up sets the handle's TIMEOUT bit.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "tc_util.h"
#include <type_traits>

namespace {

using namespace tc;

constexpr int D = AATC_D;
constexpr int EB = 128;                 // tokens per block (MMA M)
constexpr int NGRP = 4;                 // epilogue groups, one tensor-memory accumulator each
constexpr int EPI = 4 * NGRP;           // epilogue warps (4 per group: one per tensor-memory lane quarter)
constexpr int ETHREADS = (EPI + 2) * 32;   // + MMA warp + TMA warp
constexpr uint32_t XBYTES = EB * D * 2; // 32 KB per x tile
constexpr uint32_t TBYTES = 3 * D * D * 2;

__device__ __forceinline__ int key_word_pos(int i, int w, int W)
{
    const int r = w >> 2, nr = min(4, W - 4 * r), ii = i & 15;
    return 16 * W * (i >> 4) + 64 * r + (ii >> 1) * 2 * nr + 2 * (w - 4 * r) + (ii & 1);
}

struct EncArgs {
    int B, H, L_new, start_pos, Wk, Wv, nblk, n_items;   // Wk / Wv: record words of keys / values
    const int32_t *row_start;   // [B] first position of each row, or NULL: start_pos
    CacheMap map;               // contiguous or paged cache
    const EncCol *cols;     // [H][2][D]
    const uint32_t *wfix;   // [H][2][ENC_MAX_WORDS]
    uint32_t *kp, *vp;
    uint32_t *status;
};

// ES x stages: a tile's TMA load is issued as soon as the MMAs of the item ES
// back have finished with its stage, so about ES - 1 items of tensor work
// cover the load's latency
template <int ES>
__global__ void __launch_bounds__(ETHREADS, 1)
    k_encode_tc(const __grid_constant__ CUtensorMap mxk, const __grid_constant__ CUtensorMap mxv,
                const __grid_constant__ CUtensorMap mt, EncArgs a)
{
    extern __shared__ unsigned char sm_raw[];
    // 1024-byte aligned in the shared window; derived from sm_raw by pointer arithmetic so that
    // every access through it compiles to a shared-memory instruction
    unsigned char *sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
    unsigned char *Ts = sm;                              // 3 splits x 2 k-halves x 16 KB
    unsigned char *Xs = Ts + TBYTES;                     // ES x 32 KB
    uint32_t *Rs = reinterpret_cast<uint32_t *>(Xs + ES * XBYTES);   // NGRP x 128 x max(Wk, Wv) words (tiled)
    const int Wmax = a.Wk > a.Wv ? a.Wk : a.Wv;
    EncCol *cols_s = reinterpret_cast<EncCol *>(Rs + NGRP * EB * Wmax);  // [NGRP][D]
    uint32_t *wfix_s = reinterpret_cast<uint32_t *>(cols_s + NGRP * D);    // [NGRP][ENC_MAX_WORDS]
    __shared__ __align__(8) uint64_t x_full[ES], x_empty[ES], t_full, mma_done[NGRP], d_empty[NGRP];
    __shared__ uint32_t tmem_base;
    __shared__ int s_fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // a dependent decode launch may start its prologue (it waits for this grid
    // before reading the cache)
    asm volatile("griddepcontrol.launch_dependents;");
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(NGRP * D));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == EPI * 32) {
        for (int s = 0; s < ES; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&x_empty[s], 1);
        }
        mbar_init(&t_full, 1);
        for (int g = 0; g < NGRP; ++g) {
            mbar_init(&mma_done[g], 1);
            mbar_init(&d_empty[g], 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_fail = 0;
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = tmem_base;

    const int per_ht = a.B * a.nblk;
    const int i0 = (int)((long long)blockIdx.x * a.n_items / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * a.n_items / gridDim.x);
    const int count = i1 - i0;

    if (warp == EPI + 1) {
        if (lane == 0 && count > 0) {
            // ------------------------------------------------ x-tile loads
            // item m goes into stage m % ES once the MMAs of item m - ES are done with it
            bool ok = true;
            for (int m = 0; m < count && ok; ++m) {
                const int s = m % ES;
                if (m >= ES) ok = mbar_wait1(&x_empty[s], (uint32_t)((m / ES - 1) & 1));
                if (!ok || *(volatile int *)&s_fail) break;
                const int item = i0 + m, ht = item / per_ht, rem = item % per_ht;
                const int b = rem / a.nblk, blk = rem % a.nblk, h = ht >> 1, t = ht & 1;
                const int row = (b * a.H + h) * a.L_new + blk * EB;
                const CUtensorMap *map = t ? &mxv : &mxk;
                mbar_expect(&x_full[s], XBYTES);
                tma2d(Xs + s * XBYTES, map, 0, row, &x_full[s]);
                tma2d(Xs + s * XBYTES + XBYTES / 2, map, 64, row, &x_full[s]);
            }
            if (!ok) {
                atomicOr(a.status, AATC_DEV_TIMEOUT);
                s_fail = 1;
            }
        }
    } else if (warp == EPI) {
        if (lane == 0 && count > 0) {
            // ------------------------------------------------ T loads + MMA issue
            // item n: x stage n % ES, accumulator (and epilogue group) n % NGRP
            bool ok = true;
            int ht_loaded = -1, t_uses = 0;
            for (int n = 0; n < count && ok; ++n) {
                const int item = i0 + n, ht = item / per_ht;
                if (ht != ht_loaded) {
                    // the MMAs reading the old T are done once the previous item's commit arrived
                    if (n > 0)
                        ok = ok && mbar_wait1(&mma_done[(n - 1) % NGRP], (uint32_t)(((n - 1) / NGRP) & 1));
                    mbar_expect(&t_full, TBYTES);
                    for (int sp = 0; sp < 3; ++sp)
                        for (int kh = 0; kh < 2; ++kh)
                            tma2d(Ts + (sp * 2 + kh) * (XBYTES / 2), &mt, kh * 64, (ht * 3 + sp) * D, &t_full);
                    ok = ok && mbar_wait1(&t_full, (uint32_t)(t_uses & 1));
                    ++t_uses;
                    ht_loaded = ht;
                }
                const int s = n % ES, g = n % NGRP;
                ok = ok && mbar_wait1(&x_full[s], (uint32_t)((n / ES) & 1));
                // the accumulator is free once its group read the item NGRP back
                if (n >= NGRP) ok = ok && mbar_wait1(&d_empty[g], (uint32_t)(((n / NGRP) - 1) & 1));
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint32_t xa = smem_u32(Xs + s * XBYTES), ta = smem_u32(Ts);
                const uint32_t dcol = tmem + g * D;
#pragma unroll
                for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t koff = (ks >> 2) * (XBYTES / 2) + (ks & 3) * 32;
                        mma_bf16(dcol, desc_sw128(xa + koff), desc_sw128(ta + sp * XBYTES + koff),
                                 (uint32_t)(sp > 0 || ks > 0));
                    }
                mma_commit(&mma_done[g]);
                mma_commit(&x_empty[s]);
            }
            if (!ok) {
                atomicOr(a.status, AATC_DEV_TIMEOUT);
                s_fail = 1;
            }
        }
    } else if (warp < EPI) {
        // ---------------------------------------------------- epilogue groups
        const int g = warp >> 2, wq = warp & 3;   // group, tensor-memory lane quarter
        const int gt = wq * 32 + lane;             // thread in group = token in block = lane
        const int bar_id = 1 + g;
        EncCol *cols = cols_s + g * D;
        uint32_t *wfix = wfix_s + g * ENC_MAX_WORDS;
        uint32_t *R = Rs + g * EB * Wmax;
        int ht_cols = -1;
        for (int n = g; n < count; n += NGRP) {
            const int item = i0 + n, ht = item / per_ht, rem = item % per_ht;
            const int b = rem / a.nblk, blk = rem % a.nblk, h = ht >> 1, t = ht & 1;
            const int W = t ? a.Wv : a.Wk;   // the item's tensor's record words
            if (ht != ht_cols) {
                asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(128));
                for (int e = gt; e < D; e += 128) cols[e] = a.cols[(size_t)ht * D + e];
                if (gt < ENC_MAX_WORDS) wfix[gt] = a.wfix[(size_t)ht * ENC_MAX_WORDS + gt];
                asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(128));
                ht_cols = ht;
            }
            const bool ok = mbar_wait1(&mma_done[g], (uint32_t)((n / NGRP) & 1));
            if (!ok || *(volatile int *)&s_fail) {
                if (!ok) atomicOr(a.status, AATC_DEV_TIMEOUT);
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;");
            const int tl = gt >> 5, ii = gt & 31;
            uint32_t *Rt = R + tl * 32 * W;
            uint16_t *Rt16 = reinterpret_cast<uint16_t *>(Rt);
            // key word w of token ii sits at Rk + 64 r + 2 (w - 4 r) + kb 2 n_r, r = w / 4 and
            // n_r = min(4, W - 4 r) the words of row group r (the tiled layout)
            uint32_t *Rk = Rt + 16 * W * (ii >> 4) + (ii & 1);
            const int kb = (ii & 15) >> 1;
            float fin = 0.f;
            uint32_t lo = 0;
            int w = 0;
            const uint32_t row_addr = tmem + ((uint32_t)(wq * 32) << 16) + g * D;
            // Pruned channels come last in record order with a zero range: they add no
            // bits.  A non-finite input makes every coefficient non-finite (T is dense),
            // so two coefficients per token are checked.  Eight coefficients are
            // quantized at a time (independent chains; their column constants held in
            // registers), then added into the record word, a word leaving for the
            // staging buffer wherever the column marks a word end.
            auto quantize16 = [&](const uint32_t (&r)[16], int c0, auto tk) {
                constexpr int TT = decltype(tk)::value;
#pragma unroll
                for (int h8 = 0; h8 < 16; h8 += 8) {
                    int4 cw[8];   // inv, off, top, mul
#pragma unroll
                    for (int q = 0; q < 8; ++q) cw[q] = *reinterpret_cast<const int4 *>(&cols[c0 + h8 + q]);
                    uint32_t uq[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float c = __uint_as_float(r[h8 + q]);
                        float v = fmaf(c, __int_as_float(cw[q].x), __int_as_float(cw[q].y));
                        v = fminf(fmaxf(v, 0.f), fabsf(__int_as_float(cw[q].z)));
                        // adding 1.5 * 2^23 rounds to the nearest integer, ties to even
                        uq[q] = __float_as_uint(v + 12582912.f);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t mul = (uint32_t)cw[q].w, u = uq[q];
                        lo = u * mul + lo;
                        if (cw[q].z < 0) {   // the word ends with this code
                            lo -= wfix[w];
                            if constexpr (TT == 0) {
                                const int r4 = w >> 2;
                                Rk[56 * r4 + 2 * w + kb * 2 * min(4, a.Wk - 4 * r4)] = lo;
                            } else {
                                Rt16[64 * w + ii] = (uint16_t)lo;   // half-words 2w, 2w+1 of token ii
                                Rt16[64 * w + 32 + ii] = (uint16_t)(lo >> 16);
                            }
                            lo = __umulhi(u, mul);   // the part past the word
                            ++w;
                        }
                    }
                }
            };
            // one 16-column load in flight per warp at a time (a second buffer
            // doubles the unrolled code and costs more in instruction fetch);
            // the loop is compiled once for keys and once for values, so that
            // the word placement is fixed in each
            uint32_t ra[16];
            auto run = [&](auto tk) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 16) {
                    tmem_ld16(row_addr + c0, ra);
                    tmem_wait_ld(ra);
                    if (c0 == 0) fin = __uint_as_float(ra[0]) + __uint_as_float(ra[1]);
                    quantize16(ra, c0, tk);
                }
            };
            if (t == 0) run(std::integral_constant<int, 0>{});
            else run(std::integral_constant<int, 1>{});
            asm volatile("tcgen05.fence::before_thread_sync;");
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_empty[g]);
            const int tok = blk * EB + gt;
            if (!(fabsf(fin) <= 3.4e38f) && tok < a.L_new) atomicOr(a.status, AATC_DEV_NONFINITE);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // staging -> bulk store
            asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(128));
            // ---- store the block's records: a full block starting on a tile
            // boundary leaves by bulk stores (one for its 4 tiles when they are
            // contiguous, else one per tile), anything else token by token
            uint32_t *out = t ? a.vp : a.kp;
            const int p0 = (a.row_start ? a.row_start[b] : a.start_pos) + blk * EB;
            const int ntok = min(EB, a.L_new - blk * EB);
            bool range = false;
            if (ntok == EB && (p0 & 31) == 0 && p0 >= 0) {
                if (gt < EB / 32) {   // thread gt: tile gt of the block
                    const long long tw = cache_tile_word(a.map, b, h, a.H, W, (p0 >> 5) + gt);
                    if (tw < 0) {
                        range = true;
                    } else if (!a.map.table) {
                        if (gt == 0)
                            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(out + tw),
                                         "r"(smem_u32(R)), "r"((uint32_t)(EB * W * 4))
                                         : "memory");
                    } else {
                        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(out + tw),
                                     "r"(smem_u32(R + gt * 32 * W)), "r"((uint32_t)(32 * W * 4))
                                     : "memory");
                    }
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    // the group writes this staging buffer again with its next item
                    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                }
            } else if (t == 0) {
                // partial block: per-token words (keys)
                for (int e = gt; e < ntok * W; e += 128) {
                    const int ti = e / W, ww = e % W, pos = p0 + ti;
                    const long long tw = cache_tile_word(a.map, b, h, a.H, W, pos >> 5);
                    if (tw < 0) { range = true; continue; }
                    out[tw + key_word_pos(pos & 31, ww, W)] = R[(ti >> 5) * 32 * W + key_word_pos(ti & 31, ww, W)];
                }
            } else {
                // partial block: per-token half-words (values)
                const uint16_t *R16 = reinterpret_cast<const uint16_t *>(R);
                uint16_t *o16 = reinterpret_cast<uint16_t *>(out);
                for (int e = gt; e < ntok * 2 * W; e += 128) {
                    const int ti = e / (2 * W), q = e % (2 * W), pos = p0 + ti;
                    const long long tw = cache_tile_word(a.map, b, h, a.H, W, pos >> 5);
                    if (tw < 0) { range = true; continue; }
                    const uint16_t hw = R16[2 * ((ti >> 5) * 32 * W + 16 * q + ((ti & 31) >> 1)) + (ti & 1)];
                    o16[2 * (tw + 16 * q + ((pos & 31) >> 1)) + (pos & 1)] = hw;
                }
            }
            if (range) atomicOr(a.status, AATC_DEV_RANGE);
            asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(128));
        }
        if (gt < EB / 32) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NGRP * D));
}

// T3 (three bf16 terms of T, rows in record order) and the epilogue columns
__global__ void k_enc_build(const double *__restrict__ T_k, const double *__restrict__ T_v,
                            const float *__restrict__ bk32, const float *__restrict__ bv32,
                            const CodecTables *__restrict__ tabs, const HeadPlan *__restrict__ plans,
                            __nv_bfloat16 *__restrict__ T3, EncCol *__restrict__ cols, uint32_t *__restrict__ wfix)
{
    const int h = blockIdx.x, t = blockIdx.y, n = blockIdx.z, k = threadIdx.x;
    const HeadPlan &pl = plans[h * 2 + t];
    const CodecTables &tb = tabs[h * 2 + t];
    const int j = n < pl.n_coded ? pl.order[n] : -1;
    const double *T = (t ? T_v : T_k) + (size_t)h * D * D;
    const double x = j >= 0 ? T[(size_t)j * D + k] : 0.0;
    const __nv_bfloat16 a1 = __double2bfloat16(x);
    const double r1 = x - (double)__bfloat162float(a1);
    const __nv_bfloat16 a2 = __double2bfloat16(r1);
    const double r2 = r1 - (double)__bfloat162float(a2);
    const __nv_bfloat16 a3 = __double2bfloat16(r2);
    __nv_bfloat16 *dst = T3 + (((size_t)(h * 2 + t) * 3) * D + n) * D + k;
    dst[0] = a1;
    dst[(size_t)D * D] = a2;
    dst[(size_t)2 * D * D] = a3;
    if (k == 0) {
        EncCol c;
        if (j >= 0) {
            const float bias = (t ? bv32 : bk32)[h * D + j];
            c.inv = tb.inv_step[j];
            c.off = fmaf(-bias, tb.inv_step[j], tb.mid[j]);
            int nb = 0;   // bit position of column n in its record word
            for (int m = 0; m < n; ++m) nb += tb.bits[pl.order[m]];
            nb &= 31;
            c.top = (nb + tb.bits[j] >= 32) ? -tb.top[j] : tb.top[j];   // top >= 1 for a coded channel
            c.mul = 1u << nb;
        } else {
            c.inv = 0.f;
            c.off = 0.f;
            c.top = 0.f;
            c.mul = 0u;
        }
        cols[(size_t)(h * 2 + t) * D + n] = c;
    }
    if (n == 0 && k < ENC_MAX_WORDS) {
        // word k's constant: the 0x4B400000 parts of the codes that start in it,
        // shifted to their positions (mod 2^32), plus the high parts of those
        // that end past the word before it
        uint32_t fix = 0;
        int pos = 0;
        for (int m = 0; m < pl.n_coded; ++m) {
            const int b = tb.bits[pl.order[m]], wd = pos >> 5, sh = pos & 31;
            const unsigned long long part = 0x4B400000ull << sh;
            if (wd == k) fix += (uint32_t)part;
            if (wd + 1 == k && sh + b >= 32) fix += (uint32_t)(part >> 32);
            pos += b;
        }
        wfix[(h * 2 + t) * ENC_MAX_WORDS + k] = fix;
    }
}

// The driver's tensor-map encoder, found through the runtime so that the
// library does not link against the driver library itself.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

// bf16 rows of `inner` elements (row stride inner * 2 bytes), boxes of 64 x 128
// with 128-byte swizzle (the K-major operand tile of the kind::f16 MMAs).
bool encode_tma(CUtensorMap *m, const void *base, unsigned long long inner, unsigned long long rows)
{
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t enc_smem(int W, int es)
{
    return 1024 + TBYTES + es * XBYTES + NGRP * (size_t)EB * W * 4 + NGRP * D * sizeof(EncCol) +
           NGRP * ENC_MAX_WORDS * sizeof(uint32_t);
}

// largest dynamic shared memory a CTA of this device may opt into
int smem_optin_enc()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        n = (cudaGetDevice(&dev) == cudaSuccess &&
             cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess && v > 0)
                ? v
                : 232448;
    }
    return n;
}

int sm_count_enc()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        n = (cudaGetDevice(&dev) == cudaSuccess &&
             cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
                ? v
                : 148;
    }
    return n;
}

}  // namespace

bool tma_map_bf16(void *map128, const void *base, unsigned long long inner, unsigned long long rows)
{
    static_assert(sizeof(CUtensorMap) <= 128, "tensor map storage");
    return encode_tma(reinterpret_cast<CUtensorMap *>(map128), base, inner, rows);
}

aatc_status enc_build(aatc_calib *h, cudaStream_t s)
{
    k_enc_build<<<dim3(h->Hkv, 2, D), D, 0, s>>>(h->T_k, h->T_v, h->bk32, h->bv32, h->tab, h->plan,
                                                 (__nv_bfloat16 *)h->T3, h->enc_cols, h->enc_wfix);
    AATC_CUDA(cudaGetLastError());
    CUtensorMap m;
    h->tmap_ok = encode_tma(&m, h->T3, D, (unsigned long long)h->Hkv * 2 * 3 * D);
    static_assert(sizeof(CUtensorMap) <= sizeof(h->tmap_T3), "tensor map storage");
    memcpy(h->tmap_T3, &m, sizeof(m));
    return AATC_OK;
}

aatc_status encode_tc_run(const aatc_calib *h, const void *k, const void *v, int B, int L_new, int start_pos,
                          const int32_t *row_start, const CacheMap &map, uint32_t *kp, uint32_t *vp, cudaStream_t s)
{
    const unsigned long long rows = (unsigned long long)B * h->Hkv * L_new;
    CUtensorMap mk, mv, mt;
    if (!encode_tma(&mk, k, D, rows) || !encode_tma(&mv, v, D, rows))
        return aatc_fail(AATC_ERR_CUDA, "cuTensorMapEncodeTiled failed for the encoder inputs");
    memcpy(&mt, h->tmap_T3, sizeof(mt));
    EncArgs a;
    a.B = B;
    a.H = h->Hkv;
    a.L_new = L_new;
    a.start_pos = start_pos;
    a.row_start = row_start;
    a.map = map;
    a.Wk = h->Wk;
    a.Wv = h->Wv;
    a.nblk = (L_new + EB - 1) / EB;
    a.n_items = h->Hkv * 2 * B * a.nblk;
    a.cols = h->enc_cols;
    a.wfix = h->enc_wfix;
    a.kp = kp;
    a.vp = vp;
    a.status = h->status;
    // three x stages when they fit beside the staging buffers (1 KB left for the
    // kernel's static shared variables), else two
    const int W = h->Wk > h->Wv ? h->Wk : h->Wv;
    const bool three = enc_smem(W, 3) + 1024 <= (size_t)smem_optin_enc();
    const size_t smem = enc_smem(W, three ? 3 : 2);
    const void *kern = three ? (const void *)k_encode_tc<3> : (const void *)k_encode_tc<2>;
    aatc_status st = kernel_smem_limit(kern, smem);
    if (st != AATC_OK) return st;
    int grid = sm_count_enc();
    if (grid > a.n_items) grid = a.n_items;
    if (three)
        k_encode_tc<3><<<grid, ETHREADS, smem, s>>>(mk, mv, mt, a);
    else
        k_encode_tc<2><<<grid, ETHREADS, smem, s>>>(mk, mv, mt, a);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

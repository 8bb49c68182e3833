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
//   k_decode_fast   one CTA per SM, each over a contiguous range of 32-token
//                   tiles of one (batch row, KV head, head group).  It
//                   computes q' for the head group and expands it to one fp16
//                   hi/lo weight per record piece in mma.sync B-fragment
//                   order; each warp streams its own tiles into shared memory
//                   with cp.async.bulk (evict-first in L2), unpacks pieces
//                   with one AND per two fp16 operands, runs scores and P.V on
//                   mma.sync (fp16 hi/lo operands, fp32 accumulation) with an
//                   exp2 online softmax; the warps merge by log-sum-exp.  A
//                   unit split over several CTAs leaves one partial per split
//                   (in the transform domain) and the split counted in last
//                   merges them; either way Uv is applied once per head, by
//                   one CTA, and the output written.
// General path (any shape): one thread per token, codes read by offset.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <atomic>
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
constexpr int PSTRIDE = 40;      // halfs per row of the per-warp P buffer (32 tokens + pad)
constexpr int FAST_MAX_W = 16;
constexpr int PROW = 4 + D;      // floats per partial: m, l, 2 pad, acc[D] (acc 16-byte aligned)
constexpr int PSH = 6;           // P operands carry p * 2^PSH
constexpr float RESCALE_T = 8.f; // the running maximum is raised once a score exceeds it by this (log2)
// Workspace of a call with several splits per unit: split counters (one per
// unit; units number fewer than the CTAs, so at most MAX_COUNTED) at offset 0,
// where every call finds them, then the partial slots.
constexpr int MAX_COUNTED = 256;
constexpr int MERGE_MIN_SLOTS = 8;    // the merge stages at least this many partial slots at a time
constexpr int MERGE_LD = 8;           // ... and at most MERGE_LD float4 loads per thread per chunk
constexpr int SCR_CF = 256;      // epilogue: c [HPG][D] starts this many floats into the scratch (after the warp maxima and sums)
constexpr int QHS = D + 8;       // halfs per row of the fp16 B operands of the matrix products (padded: no bank conflicts)
// appender CTAs (fused append): tokens per row, padded row of T, record words
constexpr int APP_MAX = 4;
constexpr int APP_PAIRS = 4;      // (KV head, row) pairs per appender CTA at most
constexpr int APP_TILES = 48;     // tiles per split per appender pair for the fused kernel to pay
constexpr int APP_TAILS = 64;     // units an appender may have to finish (APP_PAIRS x head groups)
constexpr int APP_RW = FAST_MAX_W;
constexpr size_t APP_TT = (size_t)2 * D * D * 4;   // the two transposed transforms, in the stage region
constexpr size_t APP_PB = (size_t)2 * APP_MAX * D * 4 + 8 * APP_MAX * 4 + (size_t)2 * APP_MAX * D * 2 +
                          (size_t)2 * APP_MAX * APP_RW * 4;   // tokens, scores, codes, records, in the P buffers
constexpr size_t WS_COUNTERS = MAX_COUNTED * sizeof(unsigned);

// Work split: every (batch row, KV head, head group) is a "unit" of
// n_tiles = ceil(L/32) tiles, cut into S = max(1, resident CTAs / units)
// equal contiguous ranges; CTA (unit u, split s) streams range s of unit u
// and leaves partial slot s.
struct FastGeom {
    int NT;          // 8-column n-tiles (each: 4 query heads x hi/lo)
    int HPG;         // query heads per head group (4 NT)
    int HG;          // head groups per KV head
    int GMAX;        // value groups the kernel variant holds (>= groups)
    int FW;          // warps per CTA
    int FST;         // tiles in flight per warp
    int rows;        // key rows of 4 record words
    int groups;      // value groups of 8 half-words
    int KP;          // key pieces per byte the plan reads (4 or 8)
    int ksteps;      // KP rows
    int n_tiles;     // tiles per unit
    int units;       // B * Hkv * HG
    int S;           // splits (CTAs, partial slots) per unit
    int tiles_per;   // tiles per split
    int n_app;       // appender CTAs after the splits' (fused append; 0 otherwise)
    bool fuse_pays;  // fused append: the appenders finish inside the splits' time
    int grid;        // CTAs: units * S + n_app
    size_t stage_bytes, stage_region, smem, ws_total;
    bool single;     // one split per unit: the split kernel writes the output itself
};

// Shared memory of k_decode_fast, in carve order.
struct FastSmem {
    size_t stages, mat, blob, qtab, pbuf, mbar, scr, total;
};

// Wkv = W_K + W_V: words of one token's key and value records together.
FastSmem fast_smem_layout(int FW, int FST, int Wkv, int NT, int ksteps, int groups)
{
    FastSmem m;
    const int HPG = 4 * NT;
    const size_t tiles = (size_t)FW * FST * 128 * Wkv;
    // epilogue in the stage region: the warps' piece sums (packed when a warp's
    // own stages are too small), later the unit's partial slots (merge)
    size_t epi_region = (size_t)FW * 64 * groups * (HPG + 1) * 4;
    if (epi_region < (size_t)MERGE_MIN_SLOTS * HPG * PROW * 4) epi_region = (size_t)MERGE_MIN_SLOTS * HPG * PROW * 4;
    m.stages = tiles > epi_region ? tiles : epi_region;
    m.mat = (size_t)D * D * 4;   // A_k, then Uv: fp16 hi and lo planes
    m.blob = sizeof(DecBlob);
    m.qtab = (size_t)ksteps * NT * 32 * 8;
    m.pbuf = (size_t)FW * 8 * NT * PSTRIDE * 2;
    m.mbar = (((size_t)FW * FST + 2) * 8 + 15) & ~(size_t)15;
    const size_t bop = (size_t)NT * 8 * QHS * 2;                     // fp16 B operand: [NT][8][QHS]
    const size_t pro = (size_t)HPG * D * 4 + bop;                    // q', then the query rows
    const size_t epi = ((size_t)SCR_CF + (size_t)HPG * D) * 4 + bop;  // warp maxima and sums, c, then c as fp16 hi/lo
    m.scr = pro > epi ? pro : epi;
    m.total = m.stages + m.mat + m.blob + m.qtab + m.pbuf + m.mbar + m.scr;
    return m;
}

int fast_ctas_per_sm(int GMAX, int NT, int FW, size_t smem);
int sm_limit_bytes();

FastGeom fast_geom(const aatc_calib *h, int B, int L)
{
    FastGeom f;
    f.NT = h->G <= 4 ? 1 : 2;
    f.HPG = 4 * f.NT;
    f.HG = (h->G + f.HPG - 1) / f.HPG;
    f.rows = (h->Wk + 3) / 4;
    f.groups = (2 * h->Wv + 7) / 8;
    f.GMAX = f.groups <= 2 ? 2 : (f.groups <= 3 ? 3 : 4);
    f.FW = f.NT == 2 ? 12 : 16;
    f.KP = h->kpieces == AATC_KEY_PIECES ? AATC_KEY_PIECES : AATC_PIECES;
    f.ksteps = f.KP * f.rows;
    f.FST = 3;
    FastSmem m = fast_smem_layout(f.FW, f.FST, h->Wk + h->Wv, f.NT, f.ksteps, f.groups);
    if (m.total > (size_t)sm_limit_bytes()) {
        f.FST = 2;
        m = fast_smem_layout(f.FW, f.FST, h->Wk + h->Wv, f.NT, f.ksteps, f.groups);
    }
    f.smem = m.total;
    f.stage_region = m.stages;
    f.stage_bytes = (size_t)128 * (h->Wk + h->Wv);
    f.n_tiles = L > 0 ? (L + TILE - 1) / TILE : 0;
    f.units = B * h->Hkv * f.HG;
    const int per_sm = fast_ctas_per_sm(f.GMAX, f.NT, f.FW, f.smem);
    const int C = sm_count() * per_sm;
    f.S = C / f.units > 1 ? C / f.units : 1;
    if (f.S > f.n_tiles) f.S = f.n_tiles > 0 ? f.n_tiles : 1;
    // A unit with a single split finishes in its own CTA (no combine kernel, no workspace).
    f.single = f.n_tiles > 0 && f.S == 1;
    f.tiles_per = f.n_tiles > 0 ? (f.n_tiles + f.S - 1) / f.S : 1;
    f.S = f.n_tiles > 0 ? (f.n_tiles + f.tiles_per - 1) / f.tiles_per : 1;
    f.ws_total = f.single ? 0 : WS_COUNTERS + ((((size_t)f.units * f.S * f.HPG * PROW * 4) + 255) & ~(size_t)255);
    f.n_app = 0;
    f.grid = f.units * f.S;
    return f;
}

// Fused append + decode: the splits of a plain decode over the L_old cached
// tokens and appender CTAs on the SMs left over, each taking a contiguous run
// of the (KV head, row) pairs; one more partial slot per unit for the new
// tokens.  An appender takes about 5 us per pair, so it must not outlast the
// splits: with fewer SMs left over than pairs, the appenders keep several
// pairs each only when the splits have at least 64 tiles each per pair (about
// 8 us); otherwise the splits give up SMs so that every pair has an appender,
// if at least two splits per unit remain (n_app = 0: the shape is not fused).
// S = 0 (no split CTAs) when L_old = 0.
FastGeom fast_geom_append(const aatc_calib *h, int B, int L_old)
{
    FastGeom f = fast_geom(h, B, L_old > 0 ? L_old : 1);
    f.n_tiles = (L_old + TILE - 1) / TILE;
    const int per_sm = fast_ctas_per_sm(f.GMAX, f.NT, f.FW, f.smem);
    const int C = sm_count() * per_sm, pairs = B * h->Hkv;
    f.fuse_pays = true;
    if (f.n_tiles == 0) {
        f.S = 0;
        f.tiles_per = 1;
        f.n_app = min(pairs, C);
    } else {
        const int left = C - f.units * f.S;
        const int ppa = left > 0 ? (pairs + left - 1) / left : pairs;
        if (left >= pairs) {
            f.n_app = pairs;
            f.fuse_pays = f.tiles_per >= APP_TILES;
        } else if (left > 0 && f.tiles_per >= APP_TILES * ppa) {
            f.n_app = left;
        } else {
            const int S2 = min((C - pairs) / f.units, f.n_tiles);
            f.n_app = 0;
            if (S2 >= 2) {
                f.tiles_per = (f.n_tiles + S2 - 1) / S2;
                f.S = (f.n_tiles + f.tiles_per - 1) / f.tiles_per;
                f.n_app = pairs;
                f.fuse_pays = f.tiles_per >= APP_TILES;
            }
        }
    }
    f.grid = f.units * f.S + f.n_app;
    f.single = false;   // every unit has the appenders' slot: partials and counters always
    f.ws_total = WS_COUNTERS + ((((size_t)f.units * (f.S + 1) * f.HPG * PROW * 4) + 255) & ~(size_t)255);
    return f;
}

// aatc_set_fused_step: 0 never fuse, 1 when it pays (default), 2 whenever the shape fits
std::atomic<int> g_fuse_mode{1};

// The appender CTAs need their staging in the stage region, the unit counters
// and at most APP_MAX new tokens per row.
// and at most APP_MAX new tokens per row.  The fused kernel pays where the
// splits' merge is there anyway (several splits per unit, or no cached tokens)
// and each appender takes at most APP_PAIRS pairs, so that the appenders finish
// inside the splits' time.
bool fused_append_fits(const aatc_calib *h, const FastGeom &f, int B, int n_new)
{
    const size_t pbuf = (size_t)f.FW * 8 * f.NT * PSTRIDE * 2;
    const int mode = g_fuse_mode.load(std::memory_order_relaxed);
    return n_new >= 1 && n_new <= APP_MAX && f.stage_region >= APP_TT / 2 && pbuf >= APP_PB && f.units <= MAX_COUNTED &&
           (long)B * f.HG <= 65535 && f.S != 1 && f.n_app > 0 && (long)B * h->Hkv <= (long)APP_PAIRS * f.n_app &&
           (mode == 2 || (mode == 1 && f.fuse_pays));
}

// 8 key pieces per byte are served with GQA groups up to 4 (one n-tile: the
// kernel variant with two n-tiles has no registers to spare for the masks)
bool fast_ok(const aatc_calib *h)
{
    return h->Wk <= FAST_MAX_W && h->Wv <= FAST_MAX_W && h->fast_layout &&
           (h->kpieces == AATC_PIECES || h->G <= 4);
}

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
// lane) if it did not complete within `tries` tries.
constexpr int WAIT_TRIES = 1 << 16;   // about 1.3 s
__device__ __forceinline__ bool mbar_wait(uint64_t *mb, uint32_t parity, int tries = WAIT_TRIES)
{
    const uint32_t a = smem_u32(mb);
    // each try may suspend the thread for up to ~20 us until the phase completes
    for (int it = 0; it < tries; ++it) {
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

// L2 policy for data read once per call (the packed cache): evicted first, so
// that what every call reuses -- the kernels' code, the handle's tables, the
// query and the partials -- stays in L2 while the cache streams through it.
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *mb, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(mb)), "l"(pol)
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

// d = A B with a zero accumulator passed as its own operand (no register to clear).
__device__ __forceinline__ void mma16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 2^x for x = -inf or a finite value in the normal range (hardware exp2).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Exact power of two 2^e, e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// e with 2^e <= x < 2^(e+1) for the bits of a positive normal float x, 0 for
// x = 0, clamped to [-100, 100].
__device__ __forceinline__ int pow2_exp(int bits)
{
    return bits > 0 ? max(-100, min(100, ((bits >> 23) & 255) - 127)) : 0;
}

// Tile word of record word w of token i (0..31) of a key tile of W-word records.
__device__ __forceinline__ int key_tile_word(int i, int w, int W)
{
    const int r = w >> 2, nr = min(4, W - 4 * r), ii = i & 15;
    return 16 * W * (i >> 4) + 64 * r + (ii >> 1) * 2 * nr + 2 * (w - 4 * r) + (ii & 1);
}

// mma.sync A fragments of the 16 x 16 tile (rows r0.., columns k0..) of a
// [D][D] fp16 plane stored with 16-byte chunk n of row r at chunk n ^ (r % 8).
__device__ __forceinline__ void ldsm_x4(uint32_t (&a)[4], const __half *plane, int r0, int k0, int lane)
{
    const int q = lane >> 3, r = r0 + (q & 1) * 8 + (lane & 7), ch = (k0 >> 3) + (q >> 1);
    const __half *p = plane + r * D + ((ch ^ (r & 7)) << 3);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(smem_u32(p)));
}

struct FastArgs {
    const uint32_t *kp, *vp;
    uint32_t *kw, *vw;      // the same caches, written by the appender CTAs (fused append)
    const int32_t *seq_lens;
    CacheMap map;           // contiguous or paged cache
    int L, Wk, Wv, rows, groups, Hkv, G, HG, FST, n_tiles, units, S, tiles_per;   // Wk / Wv: record words
    int S_slots;            // partial slots per unit: S, or S + 1 when appender CTAs add one
    int n_dec;              // CTAs of the decode splits (blockIdx below n_dec); the rest are appenders
    // fused append (appender CTAs): the n_new tokens of row b and KV head h
    // at positions L_old .. L_old + n_new - 1 (the splits attend the L = L_old
    // tokens before them)
    int B, n_new, L_old;
    const void *k_new, *v_new;   // [B][Hkv][n_new][D] of the handle's dtype
    const float *TT;             // [Hkv][2][D][D] transforms T_k, T_v transposed ([k][j], fp32)
    const float *bk, *bv;        // [Hkv][D] T mu (fp32)
    const CodecTables *tabs;     // [Hkv][2]
    const HeadPlan *plans;       // [Hkv][2]
    int app_one_t;               // the stage region holds one transform at a time (below 2 D^2 floats)
    uint32_t stage_region;  // bytes before the tables: the tile stages, reused by the epilogue
    int single;             // one split per unit (S = 1): finish here and write out
    float *out;             // [B][Hq][D] (single split)
    const float *vcst;      // [Hkv][D] mu_v - Uv (Delta_V o mid) (single split)
    const DecBlob *blob;    // [Hkv]
    const __half *mats;     // [Hkv][4][D][D]: A_k hi, lo; Uv hi, lo (the handle's fp16 operand planes)
    const void *q;          // [B][Hq][D] of the handle's dtype
    float *part;            // [units][S][HPG][PROW]
    unsigned *counter;      // [units] splits counted in so far (0 between calls)
    int merge_slots;        // partial slots the stage region holds at a time (the merge)
    uint32_t *status;
    int wait_tries;         // test hook: limit of the wait for the copy left unissued
    int skip_first_copy;    // test hook: CTA 0, warp 0 leaves its first tile copy unissued
};

// One CTA = one split of one unit.  Every warp streams its own tiles
// (tile ta + warp + i FW of the split) through FST shared-memory stages.
//
// Scores (per half-tile of 16 tokens): A = key pieces (rows = tokens 2g and
// 2g+1 of the half, k = record pieces), B = query weights (8 columns = 4
// heads x hi/lo fp16 parts of q'), fp32 accumulation on mma.sync.  P.V: A =
// value pieces (rows = pieces of 8 half-words), B = P (k = tokens, columns =
// heads x hi/lo fp16 parts of p * 2^PSH).  The softmax maximum is raised
// only when a score exceeds it by RESCALE_T, so p * 2^PSH stays below 2^14.
// Each tile's P.V starts from zero and is added to the running sums in
// fp32, so the tensor-core accumulation (which does not round to nearest)
// never carries more than one tile.
// WK, WV, FSTC > 0: the record widths and the pipeline depth as compile-time
// constants (the common widths: record addressing, row and group counts fold
// away, about 5-9 % of the call at 2.75 bits); 0: read from the arguments.
template <int GMAX, int NT, int FW, int KP, typename QT, bool PAGED, int WK = 0, int WV = 0, int FSTC = 0>
__global__ void __launch_bounds__(FW * 32, 1) k_decode_fast(FastArgs a)
{
    constexpr int NTH = FW * 32;
    constexpr int HPG = 4 * NT;
    asm volatile("griddepcontrol.launch_dependents;");   // the next kernel on the stream may start its prologue
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int g = lane >> 2, c = lane & 3;
    const int Wk = WK > 0 ? WK : a.Wk, Wv = WV > 0 ? WV : a.Wv;
    const int rows = WK > 0 ? (WK + 3) / 4 : a.rows, groups = WV > 0 ? (2 * WV + 7) / 8 : a.groups;
    const int FST = FSTC > 0 ? FSTC : a.FST;
    const int ksteps = rows * KP;
    const uint32_t SB = 128u * (Wk + Wv), kbytes = 128u * Wk, vbytes = 128u * Wv;   // stage = K tile, V tile

    // shared memory carve-up (as in fast_smem_layout)
    unsigned char *stage_base = smem;
    unsigned char *mat_s = smem + a.stage_region;   // A_k, then Uv: fp16 [2][D][D] (hi, lo)
    DecBlob *blob_s = reinterpret_cast<DecBlob *>(mat_s + D * D * 4);
    uint2 *qtab_s = reinterpret_cast<uint2 *>(blob_s + 1);
    __half *pbuf = reinterpret_cast<__half *>(qtab_s + ksteps * NT * 32);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(pbuf + FW * 8 * NT * PSTRIDE);   // [FW][FST], blob, mat
    float *scr = reinterpret_cast<float *>(
        reinterpret_cast<unsigned char *>(mbar) + ((((size_t)FW * FST + 2) * 8 + 15) & ~(size_t)15));
    uint64_t *blob_bar = mbar + FW * FST;
    uint64_t *mat_bar = blob_bar + 1;   // splits: phase 0 the A_k planes, phase 1 the Uv planes
    __shared__ int mxi[8], mxq[8], mxc[8];   // largest |q'|, |q|, |c| per head (float bits)
    __shared__ float cm[8], cl[8];
    float *qpa = scr;                                          // [HPG][D] q'
    __half *qh = reinterpret_cast<__half *>(scr + HPG * D);   // [NT][8][QHS]: n-tile t = heads 4t.., hi rows then lo rows
    float *cf = scr + SCR_CF;                                 // [HPG][D] c: Delta_V o channel sums
    __half *ch = reinterpret_cast<__half *>(cf + HPG * D);    // [NT][8][QHS] c as the fp16 B operand
    // q'_i = (A_k q_i) o Delta_K / sqrt(d) for the head group on mma.sync, from
    // the A_k planes in mat_s and the query rows in qh (fp16 hi + lo, head i
    // scaled by 2^(13 - e(mxq_i))); into qpa, the largest |q'_i| into mxi
    // merge of a unit's nslots partial slots at Pu, once per head: c = sum_s
    // 2^(m_s - M) c_s and l likewise, into cf, cl and mxc (zero at entry)
    auto merge_unit = [&](const float *Pu, int nslots) {
        // merge, once per head: c = sum_s 2^(m_s - M) c_s and l likewise.  The
        // unit's partial slots are contiguous: chunks of up to merge_slots of
        // them come into the stages, every thread loading its share at once
        // from L2 (ld.global.cg: no stale L1 line), one round trip per chunk;
        // thread (head i, channel j) merges from shared memory, rescaling its
        // running sums between chunks.
        constexpr int EPT = (HPG * D + NTH - 1) / NTH;
        float Mr[EPT], ar[EPT], lr[EPT];
#pragma unroll
        for (int q = 0; q < EPT; ++q) {
            Mr[q] = -INFINITY;
            ar[q] = 0.f;
            lr[q] = 0.f;
        }
        float *Ps = reinterpret_cast<float *>(stage_base);
        for (int c0 = 0; c0 < nslots; c0 += a.merge_slots) {
            const int n = min(a.merge_slots, nslots - c0);
            const int nq = n * HPG * PROW / 4;   // float4 of the chunk: at most MERGE_LD per thread
            const float4 *src4 = reinterpret_cast<const float4 *>(Pu + (size_t)c0 * HPG * PROW);
            float4 ld[MERGE_LD];   // every load of the chunk in flight at once
#pragma unroll
            for (int k = 0; k < MERGE_LD; ++k)
                if (tid + k * NTH < nq) ld[k] = __ldcg(src4 + tid + k * NTH);
#pragma unroll
            for (int k = 0; k < MERGE_LD; ++k)
                if (tid + k * NTH < nq) reinterpret_cast<float4 *>(Ps)[tid + k * NTH] = ld[k];
            __syncthreads();
#pragma unroll
            for (int q = 0; q < EPT; ++q) {
                const int e = tid + q * NTH;
                if (e >= HPG * D) break;
                const int i = e >> 7, j = e & (D - 1);
                const float *pi = Ps + i * PROW;
                const int sstep = HPG * PROW;
                float M = Mr[q];
                for (int s2 = 0; s2 < n; ++s2) M = fmaxf(M, pi[s2 * sstep]);
                const float r = Mr[q] == -INFINITY ? 0.f : ex2(Mr[q] - M);
                float a0 = ar[q] * r, a1 = 0.f, l0 = lr[q] * r, l1 = 0.f;
                int s2 = 0;
                for (; s2 + 2 <= n; s2 += 2) {
                    const float m0 = pi[s2 * sstep], m1 = pi[(s2 + 1) * sstep];
                    const float w0 = m0 == -INFINITY ? 0.f : ex2(m0 - M), w1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
                    a0 = fmaf(w0, pi[s2 * sstep + 4 + j], a0);
                    a1 = fmaf(w1, pi[(s2 + 1) * sstep + 4 + j], a1);
                    l0 = fmaf(w0, pi[s2 * sstep + 1], l0);
                    l1 = fmaf(w1, pi[(s2 + 1) * sstep + 1], l1);
                }
                if (s2 < n) {
                    const float m0 = pi[s2 * sstep];
                    const float w0 = m0 == -INFINITY ? 0.f : ex2(m0 - M);
                    a0 = fmaf(w0, pi[s2 * sstep + 4 + j], a0);
                    l0 = fmaf(w0, pi[s2 * sstep + 1], l0);
                }
                Mr[q] = M;
                ar[q] = a0 + a1;
                lr[q] = l0 + l1;
            }
            __syncthreads();   // the chunk's stage is refilled by the next one
        }
#pragma unroll
        for (int q = 0; q < EPT; ++q) {
            const int e = tid + q * NTH;
            if (e >= HPG * D) break;
            const int i = e >> 7, j = e & (D - 1);
            cf[i * D + j] = ar[q];
            if (j == 0) cl[i] = lr[q];
            float mx = fabsf(ar[q]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) atomicMax(&mxc[i], __float_as_int(mx));
        }
    };
    // out = Uv c / l + (mu_v - Uv (Delta_V o mid)) for head group hgg of (row bb,
    // KV head hh) from cf, cl and mxc, with the Uv planes landing in mat_s
    // (phase `parity` of mat_bar)
    auto apply_uv = [&](int bb, int hh, int hgg, bool fail, uint32_t parity) {
        __syncthreads();
        // ---- o = Uv c / l + (mu_v - Uv (Delta_V o mid)), once per head, on mma.sync:
        // A = Uv 2^13, B = c_i 2^(13 - ec_i) with 2^ec_i <= max |c_i| < 2^(ec_i + 1),
        // both as fp16 hi + lo parts, fp32 accumulation
        for (int e = tid; e < HPG * D; e += NTH) {
            const int i = e >> 7, k = e & (D - 1);
            const float x = cf[e] * pow2i(13 - pow2_exp(mxc[i]));
            const __half hi = __float2half_rn(x);
            const __half lo = __float2half_rn(x - __half2float(hi));
            __half *row = ch + ((i >> 2) * 8 + (i & 3)) * QHS + k;
            row[0] = hi;
            row[4 * QHS] = lo;
        }
        __syncthreads();
        if (!mbar_wait(mat_bar, parity)) fail = true;
        if (warp < 8) {   // warp w: output channels 16w .. 16w + 15
            const __half *Uh = reinterpret_cast<const __half *>(mat_s), *Ul = Uh + D * D;
            float dh[NT][4], dl[NT][4];
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t ah[4], al[4];
                ldsm_x4(ah, Uh, 16 * warp, 16 * ks, lane);
                ldsm_x4(al, Ul, 16 * warp, 16 * ks, lane);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const __half *cb = ch + (t * 8 + g) * QHS + 16 * ks + 2 * c;
                    const uint32_t b0 = *reinterpret_cast<const uint32_t *>(cb);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t *>(cb + 8);
                    if (ks == 0) {
                        mma16816_z(dh[t], ah[0], ah[1], ah[2], ah[3], b0, b1);
                        mma16816_z(dl[t], al[0], al[1], al[2], al[3], b0, b1);
                    } else {
                        mma16816(dh[t], ah[0], ah[1], ah[2], ah[3], b0, b1);
                        mma16816(dl[t], al[0], al[1], al[2], al[3], b0, b1);
                    }
                }
            }
            const int Hq = a.Hkv * a.G;
            const int r0 = 16 * warp + g, r1 = r0 + 8;
            const float u0 = a.vcst[hh * D + r0], u1 = a.vcst[hh * D + r1];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float v[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    v[q4] = dh[t][q4] + dl[t][q4];
                    v[q4] += __shfl_xor_sync(0xffffffffu, v[q4], 2);
                }
                if (c < 2) {   // columns 2c, 2c+1 (hi parts, the lo parts added): heads 4t + 2c, +1
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int i = 4 * t + 2 * c + (q4 & 1), gi = hgg * HPG + i, r = q4 < 2 ? r0 : r1;
                        const float Ls = cl[i];
                        if (gi < a.G)
                            a.out[((size_t)bb * Hq + hh * a.G + gi) * D + r] =
                                (Ls > 0.f && !fail) ? v[q4] * pow2i(pow2_exp(mxc[i]) - 26) / Ls + (q4 < 2 ? u0 : u1)
                                                      : 0.f;
                    }
                }
            }
        }
    };
    auto qprime_mma = [&](bool ok) {
        if (warp < 8) {   // warp w: channels 16w .. 16w + 15
            const __half *Ah = reinterpret_cast<const __half *>(mat_s), *Al = Ah + D * D;
            float dh[NT][4], dl[NT][4];
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t ah[4], al[4];
                ldsm_x4(ah, Ah, 16 * warp, 16 * ks, lane);
                ldsm_x4(al, Al, 16 * warp, 16 * ks, lane);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const __half *qb = qh + (t * 8 + g) * QHS + 16 * ks + 2 * c;
                    const uint32_t b0 = *reinterpret_cast<const uint32_t *>(qb);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t *>(qb + 8);
                    if (ks == 0) {
                        mma16816_z(dh[t], ah[0], ah[1], ah[2], ah[3], b0, b1);
                        mma16816_z(dl[t], al[0], al[1], al[2], al[3], b0, b1);
                    } else {
                        mma16816(dh[t], ah[0], ah[1], ah[2], ah[3], b0, b1);
                        mma16816(dl[t], al[0], al[1], al[2], al[3], b0, b1);
                    }
                }
            }
            // columns 2c, 2c+1: hi parts of heads 4t + 2c, +1 (c < 2) or their lo parts (c >= 2)
            const int j0 = 16 * warp + g, j1 = j0 + 8;
            const float k0 = blob_s->ksc[j0], k1 = blob_s->ksc[j1];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float v[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    v[q4] = dh[t][q4] + dl[t][q4];
                    v[q4] += __shfl_xor_sync(0xffffffffu, v[q4], 2);
                }
                const int i0 = 4 * t + 2 * (c & 1), i1 = i0 + 1;
                const float s0 = ok ? pow2i(pow2_exp(mxq[i0]) - 13) : 0.f;
                const float s1 = ok ? pow2i(pow2_exp(mxq[i1]) - 13) : 0.f;
                const float a00 = v[0] * k0 * s0, a10 = v[1] * k0 * s1, a01 = v[2] * k1 * s0, a11 = v[3] * k1 * s1;
                if (c < 2) {
                    qpa[i0 * D + j0] = a00;
                    qpa[i1 * D + j0] = a10;
                    qpa[i0 * D + j1] = a01;
                    qpa[i1 * D + j1] = a11;
                }
                float m0 = fmaxf(fabsf(a00), fabsf(a01)), m1 = fmaxf(fabsf(a10), fabsf(a11));
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
                    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
                }
                if (lane < 2) {
                    atomicMax(&mxi[i0], __float_as_int(m0));
                    atomicMax(&mxi[i1], __float_as_int(m1));
                }
            }
        }
    };

    // ---- this CTA: unit u, split sp, tiles [ta, tb) of the unit
    const int u = blockIdx.x / a.S, sp = blockIdx.x % a.S;
    const int b = u / (a.Hkv * a.HG), h = (u / a.HG) % a.Hkv, hg = u % a.HG;
    const int ta = sp * a.tiles_per, tb = min(ta + a.tiles_per, a.n_tiles);
    constexpr bool paged = PAGED;
    // first tile of this (row, KV head) in a contiguous cache, in tiles of 32 tokens
    const size_t slab_t = paged ? 0 : ((size_t)b * a.Hkv + h) * (size_t)(a.map.L_cap / TILE);
    uint64_t *my_mbar = mbar + warp * FST;
    unsigned char *my_stage = stage_base + (size_t)warp * FST * SB;

    // Barriers first (the init fence waits for the thread's outstanding memory
    // operations), then the copies the prologue needs, ahead of the tile burst.
    // The one-shot code here is kept short: it runs from a cold instruction cache.
    if (lane == 0) {
        for (int s = 0; s < FST; ++s) mbar_init(&my_mbar[s], 1);
        if (warp == 0) {
            mbar_init(blob_bar, 1);
            mbar_init(mat_bar, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (blockIdx.x >= a.n_dec) {
        // ======================================================== appenders
        // Appender i takes the pairs i P / n_app .. (i + 1) P / n_app - 1 of the
        // P = B H_kv (KV head, row) pairs (pair p: head p / B, row p % B), so that
        // consecutive pairs share a head and its tables stay in shared memory.
        // For each pair it encodes the n_new new tokens as the append encoder
        // does (fp32 transform, the same operation order), writes their records
        // into the cache, and leaves their attention -- in the form of a split's
        // partial -- in slot S of each of the pair's units, counting it in; the
        // last to count a unit in merges it.  No CTA waits for another.
        float *TT = reinterpret_cast<float *>(stage_base);                     // [2][D][D]: T_k, T_v as [k][j]
        float *xs = reinterpret_cast<float *>(pbuf);                           // [2][APP_MAX][D] new keys, values
        float *ssc = xs + 2 * APP_MAX * D;                                     // [HPG][APP_MAX] scores (log2 domain)
        int16_t *cod = reinterpret_cast<int16_t *>(ssc + 8 * APP_MAX);         // [2][APP_MAX][D] codes
        uint32_t *rec = reinterpret_cast<uint32_t *>(cod + 2 * APP_MAX * D);   // [2][APP_MAX][APP_RW] records
        __shared__ int s_tail[APP_TAILS], s_ntail;   // units this CTA counted in last, finished at the end
        uint64_t *t_bar = mbar;       // warp 0's first stage barrier: the transforms
        uint32_t tph = 0, bph = 0, mph = 0;   // next phases of t_bar, blob_bar and mat_bar
        bool ok = true, bad = false, range = false;
        const int Hq = a.Hkv * a.G, P = a.B * a.Hkv, n_app = gridDim.x - a.n_dec, ai = blockIdx.x - a.n_dec;
        const int p0 = (int)((long long)ai * P / n_app), p1 = (int)((long long)(ai + 1) * P / n_app);
        constexpr int QPA = (HPG * D + NTH - 1) / NTH;
        // heads whose transforms (TT), table blob and A_k planes (mat_s) are in
        // shared memory, -1 for none (a merge stages partials over TT; the Uv
        // planes replace the A_k planes)
        int hT = -1, hB = -1, hA = -1;
        auto load = [&](int hh) {   // thread 0: the copies the pair of head hh still needs
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // after the generic reads of these buffers
            if (!a.app_one_t && hh != hT) {   // (one-slot mode: each transform in turn, below)
                mbar_arrive_expect(t_bar, (uint32_t)(2 * D * D * 4));
                bulk_g2s(TT, a.TT + (size_t)hh * 2 * D * D, (uint32_t)(2 * D * D * 4), t_bar);
            }
            if (hh != hB) {
                mbar_arrive_expect(blob_bar, (uint32_t)sizeof(DecBlob));
                bulk_g2s(blob_s, a.blob + hh, (uint32_t)sizeof(DecBlob), blob_bar);
            }
            if (hh != hA) {
                mbar_arrive_expect(mat_bar, (uint32_t)(D * D * 4));
                bulk_g2s(mat_s, a.mats + (size_t)hh * 4 * D * D, (uint32_t)(D * D * 4), mat_bar);
            }
        };
        // the first pair's tables are handle data: requested ahead of the wait
        if (tid == 0) {
            s_ntail = 0;
            if (p0 < p1) load(p0 / a.B);
        }
        // the new tokens, the query and the cache may be written by the kernel before this one
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int p = p0; p < p1; ++p) {
            const int ph = p / a.B, pb = p % a.B;
            if (p > p0 && tid == 0) load(ph);
            // the pair's new keys and values
            for (int e = tid; e < 2 * a.n_new * D; e += NTH) {
                const int t = e / (a.n_new * D), r = e % (a.n_new * D);
                const QT *x = reinterpret_cast<const QT *>(t ? a.v_new : a.k_new) + ((size_t)pb * a.Hkv + ph) * a.n_new * D;
                const float xv = to_f32(x[r]);
                bad |= !isfinite(xv);
                xs[t * APP_MAX * D + r] = xv;
            }
            for (int e = tid; e < 2 * APP_MAX * APP_RW; e += NTH) rec[e] = 0u;
            __syncthreads();
            if (!a.app_one_t && ph != hT) {
                ok = mbar_wait(t_bar, tph) && ok;
                tph ^= 1u;
            }
            if (ph != hB) {
                ok = mbar_wait(blob_bar, bph) && ok;
                bph ^= 1u;
            }
            if (ph != hA) {
                ok = mbar_wait(mat_bar, mph) && ok;
                mph ^= 1u;
            }
            hT = hB = hA = ph;
            // thread (tensor, channel j): c = T x - T mu, quantized, ORed into the record;
            // both tensors at once, or (one-slot mode) keys then values, each transform
            // brought into the single slot in turn
            for (int phz = 0; phz < (a.app_one_t ? 2 : 1); ++phz) {
                if (a.app_one_t) {
                    if (phz == 1) __syncthreads();   // the key transform's last reads
                    if (tid == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        mbar_arrive_expect(t_bar, (uint32_t)(D * D * 4));
                        bulk_g2s(TT, a.TT + ((size_t)ph * 2 + phz) * D * D, (uint32_t)(D * D * 4), t_bar);
                    }
                    ok = mbar_wait(t_bar, tph) && ok;
                    tph ^= 1u;
                }
                if (a.app_one_t ? tid >= D : tid >= 2 * D) continue;
                const int tensor = a.app_one_t ? phz : tid >> 7, j = tid & (D - 1);
                const CodecTables &tb = a.tabs[ph * 2 + tensor];
                const float bias = (tensor ? a.bv : a.bk)[ph * D + j];
                const float inv = tb.inv_step[j], mid = tb.mid[j], top = tb.top[j];
                const int bits = tb.bits[j], off = a.plans[ph * 2 + tensor].off[j];
                const float *Tt = TT + (a.app_one_t ? 0 : (size_t)tensor * D * D);
                for (int n = 0; n < a.n_new; ++n) {
                    const float *xr = xs + (tensor * APP_MAX + n) * D;
                    float acc = 0.f;
#pragma unroll 8
                    for (int k = 0; k < D; ++k) acc = fmaf(Tt[k * D + j], xr[k], acc);
                    uint32_t uq = 0u;
                    if (bits > 0) {
                        float vq = fmaf(acc - bias, inv, mid);
                        vq = fminf(fmaxf(rintf(vq), 0.f), top);
                        uq = (uint32_t)vq;
                        uint32_t *rw = rec + (tensor * APP_MAX + n) * APP_RW;
                        const int sh = off & 31;
                        atomicOr(&rw[off >> 5], uq << sh);
                        if (sh + bits > 32) atomicOr(&rw[(off >> 5) + 1], uq >> (32 - sh));
                    }
                    cod[(tensor * APP_MAX + n) * D + j] = (int16_t)uq;
                }
            }
            if (a.app_one_t) hT = -1;   // the slot holds the value transform
            __syncthreads();
            // the records into the cache, placed as the encoders place them
            for (int e = tid; e < a.n_new * 3 * (Wk > Wv ? Wk : Wv); e += NTH) {
                // keys: W_k words per token; values: 2 W_v half-words per token
                const int per = 3 * (Wk > Wv ? Wk : Wv), n = e / per, r = e % per;
                const int pos = a.L_old + n;
                if (r < Wk) {
                    const long long tw = cache_tile_word(a.map, pb, ph, a.Hkv, Wk, pos >> 5);
                    if (tw < 0) range = true;
                    else a.kw[tw + key_tile_word(pos & 31, r, Wk)] = rec[n * APP_RW + r];
                } else if (r - Wk < 2 * Wv) {
                    const int jj = r - Wk;
                    const long long tw = cache_tile_word(a.map, pb, ph, a.Hkv, Wv, pos >> 5);
                    if (tw < 0) {
                        range = true;
                    } else {
                        const long long word = tw + 16 * jj + ((pos & 31) >> 1);
                        reinterpret_cast<uint16_t *>(a.vw)[2 * word + (pos & 1)] =
                            (uint16_t)(rec[(APP_MAX + n) * APP_RW + (jj >> 1)] >> (16 * (jj & 1)));
                    }
                }
            }
            const int16_t *uk = cod, *uv = cod + APP_MAX * D;
            for (int hgp = 0; hgp < a.HG; ++hgp) {
                const int uu = (pb * a.Hkv + ph) * a.HG + hgp;
                if (tid < 8) {
                    mxi[tid] = 0;
                    mxq[tid] = 0;
                }
                __syncthreads();
                // the head group's query rows as the fp16 B operand of q' (as in the splits)
                float qv[QPA];
#pragma unroll
                for (int r = 0; r < QPA; ++r) {
                    const int e = tid + r * NTH, i = e >> 7, gi = hgp * HPG + i;
                    qv[r] = (e < HPG * D && gi < a.G)
                                ? to_f32(reinterpret_cast<const QT *>(a.q)[((size_t)pb * Hq + ph * a.G + gi) * D + (e & (D - 1))])
                                : 0.f;
                    float mx = fabsf(qv[r]);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    if (lane == 0 && e < HPG * D) atomicMax(&mxq[i], __float_as_int(mx));
                }
                __syncthreads();
#pragma unroll
                for (int r = 0; r < QPA; ++r) {
                    const int e = tid + r * NTH;
                    if (e < HPG * D) {
                        const int i = e >> 7, k = e & (D - 1);
                        const float xq = qv[r] * pow2i(13 - pow2_exp(mxq[i]));
                        const __half hi = __float2half_rn(xq);
                        const __half lo = __float2half_rn(xq - __half2float(hi));
                        __half *row = qh + ((i >> 2) * 8 + (i & 3)) * QHS + k;
                        row[0] = hi;
                        row[4 * QHS] = lo;
                    }
                }
                __syncthreads();
                qprime_mma(ok);
                __syncthreads();
                // scores of the new tokens in the log2 domain, q'_i . u_n log2(e) (the splits' scale)
                for (int e = tid; e < HPG * a.n_new; e += NTH) {
                    const int i = e / a.n_new, n = e % a.n_new;
                    float sacc = 0.f;
                    for (int j = 0; j < D; ++j) sacc = fmaf(qpa[i * D + j], (float)uk[n * D + j], sacc);
                    ssc[i * APP_MAX + n] = sacc * LOG2E;
                }
                __syncthreads();
                // their partial, as a split leaves one: m_i, l_i = sum_n 2^(s_n - m_i + PSH),
                // c_ij = Delta_V,j sum_n 2^(s_n - m_i + PSH) u_nj
                float *Pg = a.part + ((size_t)uu * a.S_slots + (a.S_slots - 1)) * HPG * PROW;
                for (int e = tid; e < HPG * D; e += NTH) {
                    const int i = e >> 7, j = e & (D - 1);
                    float M = -INFINITY;
                    for (int n = 0; n < a.n_new; ++n) M = fmaxf(M, ssc[i * APP_MAX + n]);
                    float l = 0.f, cacc = 0.f;
                    for (int n = 0; n < a.n_new; ++n) {
                        const float pn = ex2(ssc[i * APP_MAX + n] - M + (float)PSH);
                        l += pn;
                        cacc = fmaf(pn, (float)uv[n * D + j], cacc);
                    }
                    Pg[i * PROW + 4 + j] = ok ? cacc * blob_s->vstep[j] : 0.f;
                    if (j < 4) Pg[i * PROW + j] = j == 0 ? (ok ? M : -INFINITY) : j == 1 ? (ok ? l : 0.f) : 0.f;
                }
                __syncthreads();
                if (tid == 0) {
                    unsigned old;
                    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.counter + uu) : "memory");
                    if (old >= (unsigned)a.S_slots) atomicOr(a.status, AATC_DEV_WORKSPACE);   // counters were not zero
                    if (old == (unsigned)(a.S_slots - 1)) {   // (read back only after the last pair)
                        a.counter[uu] = 0u;
                        if (s_ntail < APP_TAILS) s_tail[s_ntail++] = uu;
                        else atomicOr(a.status, AATC_DEV_WORKSPACE);
                    }
                }
            }
            __syncthreads();   // the next pair's copies overwrite what this one read
        }
        // the units this CTA counted in last: merge them, Uv of each head into mat_s
        // (the merge stages partials over TT)
        const int ntail = s_ntail;
        int hU = -1;   // the head whose Uv planes mat_s holds
        for (int k = 0; k < ntail; ++k) {
            const int uu = s_tail[k], hgp = uu % a.HG, ph = (uu / a.HG) % a.Hkv, pb = uu / (a.HG * a.Hkv);
            if (ph != hU) {
                if (tid == 0) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive_expect(mat_bar, (uint32_t)(D * D * 4));
                    bulk_g2s(mat_s, a.mats + ((size_t)ph * 4 + 2) * D * D, (uint32_t)(D * D * 4), mat_bar);
                }
                mph ^= 1u;
                hU = ph;
            }
            if (tid < 8) mxc[tid] = 0;
            __syncthreads();
            merge_unit(a.part + (size_t)uu * a.S_slots * HPG * PROW, a.S_slots);
            apply_uv(pb, ph, hgp, !ok, mph ^ 1u);
            __syncthreads();
        }
        if (!ok) {   // a wait gave up: its copy lands before the shared memory is given back
            mbar_wait(t_bar, tph ^ 1u);
            mbar_wait(blob_bar, bph ^ 1u);
            mbar_wait(mat_bar, mph ^ 1u);
        }
        if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, AATC_DEV_NONFINITE);
        if (range) atomicOr(a.status, AATC_DEV_RANGE);
        if (!ok && tid == 0) atomicOr(a.status, AATC_DEV_TIMEOUT);
        return;
    }
    if (tid == 0) {
        mbar_arrive_expect(blob_bar, (uint32_t)sizeof(DecBlob));
        bulk_g2s(blob_s, a.blob + h, (uint32_t)sizeof(DecBlob), blob_bar);
        mbar_arrive_expect(mat_bar, (uint32_t)(D * D * 4));
        bulk_g2s(mat_s, a.mats + (size_t)h * 4 * D * D, (uint32_t)(D * D * 4), mat_bar);
    }
    if (tid < 8) {
        mxi[tid] = 0;
        mxq[tid] = 0;
        mxc[tid] = 0;
    }
    __syncthreads();   // (the maxima are zero before any thread raises them)
    // Launched with programmatic dependent launch: everything above reads only
    // the handle; the query, the row lengths, the cache and the workspace may
    // be written by the kernel before this one on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // paged cache: lane 0 reads the block table entries of the warp's first
    // FST tiles (ent) and of its next three refills (r0, r1, r2), ahead of the
    // tile burst; each refill then reads the entry three refills ahead, since a
    // load issued behind the burst waits for the copies queued before it
    // (tiles below tb are inside the table)
    const int sh = a.map.tpb_shift;
    int ent[3] = {0, 0, 0}, r0 = 0, r1 = 0, r2 = 0;
    bool bad_blk = false;
    const int32_t *trow = paged ? a.map.table + (size_t)b * a.map.bpr : nullptr;
    if (paged && lane == 0) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int tile = ta + warp + i * FW;
            if (i < FST && tile < tb) ent[i] = trow[tile >> sh];
        }
        const int tr = ta + warp + FST * FW;
        if (tr < tb) r0 = trow[tr >> sh];
        if (tr + FW < tb) r1 = trow[(tr + FW) >> sh];
        if (tr + 2 * FW < tb) r2 = trow[(tr + 2 * FW) >> sh];
    }
    // tile index (in 32-token tiles) of a tile of this (row, KV head) in the pool
    // (block 0 for a bad entry); a tile's words start at 32 W times it
    auto pool_tile = [&](int blk, int tile) -> size_t {
        if (blk < 0 || blk >= a.map.n_blocks) {
            bad_blk = true;
            blk = 0;
        }
        return (((size_t)blk * a.Hkv + h) << sh) + (size_t)(tile & ((1 << sh) - 1));
    };
    // query rows of the head group: element e = (head e / D, k = e % D), loaded
    // as raw bits ahead of the tile burst and converted after it, so that no
    // thread waits for them before issuing its copies
    constexpr int QPER = (HPG * D + NTH - 1) / NTH;
    uint32_t qraw[QPER];
    {
        const int Hq = a.Hkv * a.G;
#pragma unroll
        for (int r = 0; r < QPER; ++r) {
            const int e = tid + r * NTH, gi = hg * HPG + (e >> 7);
            const size_t idx = ((size_t)b * Hq + h * a.G + gi) * D + (e & (D - 1));
            qraw[r] = 0u;
            if (e < HPG * D && gi < a.G) {
                if (sizeof(QT) == 2) qraw[r] = reinterpret_cast<const unsigned short *>(a.q)[idx];
                else qraw[r] = reinterpret_cast<const uint32_t *>(a.q)[idx];
            }
        }
    }
    const int len = a.seq_lens ? min(max(a.seq_lens[b], 0), a.L) : a.L;

    const uint64_t stream_pol = evict_first_policy();
    auto issue = [&](size_t tidx, int s) {   // tile tidx of the cache (K and V) into stage s
        unsigned char *dst = my_stage + s * SB;
        mbar_arrive_expect(&my_mbar[s], kbytes + vbytes);
        bulk_g2s_hint(dst, a.kp + tidx * TILE * Wk, kbytes, &my_mbar[s], stream_pol);
        bulk_g2s_hint(dst + kbytes, a.vp + tidx * TILE * Wv, vbytes, &my_mbar[s], stream_pol);
    };
    // The warp's n-th tile goes through stage n % FST and completes phase
    // n / FST of that stage's barrier.  In a contiguous cache the first tiles
    // are requested up to tb, before the row length has arrived (tiles below
    // tb are inside the cache); copies past the row's length are drained at
    // the end.  In a paged cache only tiles inside the row are requested.
    int n_issued = 0, n_done = 0;
    // test hook (aatc_test_wait_fault): this warp's first copy is never issued,
    // so its wait for it runs out (after a.wait_tries tries) and reports TIMEOUT
    const bool hook = a.skip_first_copy && blockIdx.x == 0 && warp == 0;
    int st_next = 0;          // stage of the next tile to consume
    uint32_t ph_next = 0;     // its barrier phase parity
    const int t1 = min(tb, (len + TILE - 1) / TILE);
    // first copies of stages [i0, i1): the copy engine takes requests one at
    // a time, so the issuing lane waits while the CTA's requests queue up;
    // stage 0 goes out before the query weights are built, the rest after
    auto burst = [&](int i0, int i1) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {   // FST <= 3
            const int tile = ta + warp + i * FW;
            if (i < i0 || i >= i1) continue;
            if (!paged && tile < tb) {
                if (lane == 0 && !(hook && i == 0)) issue(slab_t + (size_t)tile, i);
                ++n_issued;
            }
            if (paged && tile < t1) {
                if (lane == 0 && !(hook && i == 0)) issue(pool_tile(ent[i], tile), i);
                ++n_issued;
            }
        }
    };
    burst(0, 1);

    // ---- query weights of the head group: q' = (A_k q) o Delta_K / sqrt(d) on
    // mma.sync (A = rows of A_k, B = the query rows, both as fp16 hi + lo
    // parts scaled by powers of two; fp32 accumulation), then scaled per head
    // by a power of two S_i, split into fp16 hi/lo parts and laid out as
    // mma.sync B fragments for the tile loop.
    float sc[NT];   // log2-domain score scale of head 4t + c: 2^24 / S_i * log2(e)
    bool ok;
    {
        float *pa = qpa;
        float qv[QPER];
#pragma unroll
        for (int r = 0; r < QPER; ++r) {
            uint32_t x;   // bf16 or fp32 bits -> fp32 bits; asm volatile keeps it (the load's first use) after the burst
            if (sizeof(QT) == 2) asm volatile("shl.b32 %0, %1, 16;" : "=r"(x) : "r"(qraw[r]));
            else asm volatile("mov.b32 %0, %1;" : "=r"(x) : "r"(qraw[r]));
            qv[r] = __uint_as_float(x);
            // a warp's 32 elements belong to one head: its largest |q| per head
            float mx = fabsf(qv[r]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const int e = tid + r * NTH;
            if (lane == 0 && e < HPG * D) atomicMax(&mxq[e >> 7], __float_as_int(mx));
        }
        __syncthreads();
        // B operand: q_i 2^(13 - eq_i), 2^eq_i <= max |q_i| < 2^(eq_i + 1), as fp16 hi + lo
#pragma unroll
        for (int r = 0; r < QPER; ++r) {
            const int e = tid + r * NTH;
            if (e < HPG * D) {
                const int i = e >> 7, k = e & (D - 1);
                const float x = qv[r] * pow2i(13 - pow2_exp(mxq[i]));
                const __half hi = __float2half_rn(x);
                const __half lo = __float2half_rn(x - __half2float(hi));
                __half *row = qh + ((i >> 2) * 8 + (i & 3)) * QHS + k;
                row[0] = hi;
                row[4 * QHS] = lo;
            }
        }
        __syncthreads();
        ok = mbar_wait(mat_bar, 0);
        ok = mbar_wait(blob_bar, 0) && ok;
        qprime_mma(ok);
        __syncthreads();
        // A_k is used up: Uv comes into the same buffer for the split that
        // finishes the unit (the only one, or whichever is counted in last)
        if (tid == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect(mat_bar, (uint32_t)(D * D * 4));
            bulk_g2s(mat_s, a.mats + ((size_t)h * 4 + 2) * D * D, (uint32_t)(D * D * 4), mat_bar);
        }
        // S_i = 2^(6 - e_i) with max|q'_i| = f 2^e_i, f in [0.5, 1): weights below 2^(6 + 7)
        auto s_exp = [&](int i) -> int {
            const int bits = mxi[i];
            const int e = bits > 0 ? ((bits >> 23) & 255) - 126 : 6;
            return max(-100, min(100, 6 - e));
        };
        // B fragments: entry (kstep, n-tile t, lane) = (b0, b1), column n = 8t + lane/4 =
        // (head n/2, hi if n even else lo), k-step (r, s4 < KP) from record word 4r + lane%4,
        // slots 2 s4 (b0) and 2 s4 + 1 (b1), low half first; weight = q'_ch * 2^ex * S
        for (int en = tid; en < ksteps * NT * 32; en += NTH) {
            const int ln = en & 31, t = (en >> 5) % NT, ks = (en >> 5) / NT;
            const int r = ks / KP, s4 = ks % KP;
            const int n = 8 * t + (ln >> 2), i = n >> 1, part = n & 1;
            const int w = 4 * r + (ln & 3);
            const bool live = hg * HPG + i < a.G;
            const int se = s_exp(i);
            uint32_t o2[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int k = 2 * s4 + rr;
                float v2[2];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int sl = blob_s->kslot[w][k][half];
                    float val = 0.f;
                    if (sl >= 0 && live) val = pa[i * D + (sl & 255)] * pow2i(se + (sl >> 8) - 64);
                    const float hi = __half2float(__float2half_rn(val));
                    v2[half] = part ? val - hi : hi;
                }
                o2[rr] = pack_half2(v2[0], v2[1]);
            }
            qtab_s[en] = make_uint2(o2[0], o2[1]);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) sc[t] = LOG2E * pow2i(24 - s_exp(4 * t + c));
    }
    burst(1, FST);
    __syncthreads();

    float m_run[NT], l_run[NT];
    float acc[GMAX][4][NT][2];   // rows g / g + 8 of each value m-tile, hi + lo columns summed
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        m_run[t] = -INFINITY;
        l_run[t] = 0.f;
    }
#pragma unroll
    for (int gr = 0; gr < GMAX; ++gr)
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[gr][m4][t][0] = acc[gr][m4][t][1] = 0.f;

    __half *pw = pbuf + warp * 8 * NT * PSTRIDE;
    bool failed = !ok;
    for (int it = 0; !failed; ++it) {
        const int tile = ta + warp + it * FW;
        if (tile >= t1) break;
        const int s = st_next;
        if (!mbar_wait(&my_mbar[s], ph_next, (hook && n_done == 0) ? a.wait_tries : WAIT_TRIES)) {
            failed = true;
            break;
        }
        ++n_done;
        if (++st_next == FST) {
            st_next = 0;
            ph_next ^= 1u;
        }
        const uint32_t *Kt = reinterpret_cast<const uint32_t *>(my_stage + s * SB);
        const uint32_t *Vt = Kt + TILE * Wk;

        // ---- scores: C[hf] rows g / g+8 = tokens 16 hf + 2g / +1, columns 2c / 2c+1 =
        // head c hi / lo; one accumulator chain per half-tile, the two interleaved
        float C[2][NT][4];      // chain hf starts at row 0, k-step 0 with a zero accumulator
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (r >= rows) break;
            const int nr = min(4, Wk - 4 * r);
            uint32_t mk[2 * KP];
#pragma unroll
            for (int m4 = 0; m4 < KP / 2; ++m4) {
                const uint4 mm = *reinterpret_cast<const uint4 *>(&blob_s->kmask[4 * r + c][4 * m4]);
                mk[4 * m4] = mm.x;
                mk[4 * m4 + 1] = mm.y;
                mk[4 * m4 + 2] = mm.z;
                mk[4 * m4 + 3] = mm.w;
            }
            uint32_t x0[2], x1[2], y0[2], y1[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint2 kw = *reinterpret_cast<const uint2 *>(Kt + hf * 16 * Wk + 64 * r + g * 2 * nr + 2 * c);
                x0[hf] = kw.x;
                x1[hf] = kw.y;
                y0[hf] = kw.x >> 8;
                y1[hf] = kw.y >> 8;
            }
#pragma unroll
            for (int s4 = 0; s4 < KP; ++s4) {
                uint2 bq[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) bq[t] = qtab_s[((r * KP + s4) * NT + t) * 32 + lane];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const uint32_t sa = s4 < KP / 2 ? x0[hf] : y0[hf], sb = s4 < KP / 2 ? x1[hf] : y1[hf];
                    const uint32_t A0 = sa & mk[2 * s4], A1 = sb & mk[2 * s4];
                    const uint32_t A2 = sa & mk[2 * s4 + 1], A3 = sb & mk[2 * s4 + 1];
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (r == 0 && s4 == 0) mma16816_z(C[hf][t], A0, A1, A2, A3, bq[t].x, bq[t].y);
                        else mma16816(C[hf][t], A0, A1, A2, A3, bq[t].x, bq[t].y);
                    }
                }
            }
        }

        // ---- online softmax (log2 domain); thread owns head 4t+c of tokens 16hf+2g, +1
        const int tb0 = tile * TILE;
        const bool full = tb0 + TILE <= len;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float sv[4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                sv[2 * hf] = C[hf][t][0] + C[hf][t][1];
                sv[2 * hf + 1] = C[hf][t][2] + C[hf][t][3];
            }
            if (!full) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (tb0 + 16 * (j >> 1) + 2 * g + (j & 1) >= len) sv[j] = -INFINITY;
            }
            const float mt = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3])) * sc[t];
            if (__any_sync(0xffffffffu, mt > m_run[t] + RESCALE_T)) {
                float mw = mt;
                mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 4));
                mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 8));
                mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 16));
                const float mn = fmaxf(m_run[t], mw);
                const float alpha = ex2(m_run[t] - mn);   // 0 while nothing was seen yet
                m_run[t] = mn;
                l_run[t] *= alpha;
#pragma unroll
                for (int gr = 0; gr < GMAX; ++gr)
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {
                        acc[gr][m4][t][0] *= alpha;
                        acc[gr][m4][t][1] *= alpha;
                    }
            }
            const float mb = m_run[t] - (float)PSH;
            float p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) p[j] = ex2(fmaf(sv[j], sc[t], -mb));
            l_run[t] += (p[0] + p[1]) + (p[2] + p[3]);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                // hi/lo fp16 pair per token (hi in column 2c, lo in 2c+1)
                const __half2 hi2 = __floats2half2_rn(p[2 * hf], p[2 * hf + 1]);
                const float2 hif = __half22float2(hi2);
                const __half2 lo2 = __floats2half2_rn(p[2 * hf] - hif.x, p[2 * hf + 1] - hif.y);
                const int tau = 16 * hf + 2 * g;
                *reinterpret_cast<__half2 *>(pw + (8 * t + 2 * c) * PSTRIDE + tau) = hi2;
                *reinterpret_cast<__half2 *>(pw + (8 * t + 2 * c + 1) * PSTRIDE + tau) = lo2;
            }
        }
        __syncwarp();

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
            const uint4 mA = *reinterpret_cast<const uint4 *>(&blob_s->vmask[e][0]);
            const uint4 mB = *reinterpret_cast<const uint4 *>(&blob_s->vmask[e][4]);
            const uint32_t mv[8] = {mA.x, mA.y, mA.z, mA.w, mB.x, mB.y, mB.z, mB.w};
            const uint32_t xs[4] = {pq.x, pq.y, pq.z, pq.w};
            const uint32_t ys[4] = {pq.x >> 8, pq.y >> 8, pq.z >> 8, pq.w >> 8};
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4) {
                float ta4[NT][4];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint32_t u0 = m4 < 2 ? xs[2 * kk] : ys[2 * kk];
                    const uint32_t u1 = m4 < 2 ? xs[2 * kk + 1] : ys[2 * kk + 1];
                    const uint32_t A0 = u0 & mv[2 * m4], A1 = u0 & mv[2 * m4 + 1];
                    const uint32_t A2 = u1 & mv[2 * m4], A3 = u1 & mv[2 * m4 + 1];
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (kk == 0) mma16816_z(ta4[t], A0, A1, A2, A3, bp[kk][t].x, bp[kk][t].y);
                        else mma16816(ta4[t], A0, A1, A2, A3, bp[kk][t].x, bp[kk][t].y);
                    }
                }
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    acc[gr][m4][t][0] += ta4[t][0] + ta4[t][1];
                    acc[gr][m4][t][1] += ta4[t][2] + ta4[t][3];
                }
            }
        }
        __syncwarp();
        const int nt = tile + FST * FW;
        if (nt < t1) {
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (paged) {
                    issue(pool_tile(r0, nt), s);
                    r0 = r1;
                    r1 = r2;
                    const int nn = nt + 3 * FW;   // three refills ahead
                    r2 = nn < t1 ? trow[nn >> sh] : 0;
                } else {
                    issue(slab_t + (size_t)nt, s);
                }
            }
            ++n_issued;
        }
    }
    // copies still in flight (requested past the row's length, or left by a
    // failed wait) land before the shared memory is reused
    if (failed && lane == 0) atomicOr(a.status, AATC_DEV_TIMEOUT);
    if (bad_blk) atomicOr(a.status, AATC_DEV_RANGE);
    for (; n_done < n_issued; ++n_done) {
        // (the copy the test hook left unissued has nothing to drain)
        if (!(hook && n_done == 0) && !mbar_wait(&my_mbar[st_next], ph_next)) failed = true;
        if (++st_next == FST) {
            st_next = 0;
            ph_next ^= 1u;
        }
    }
    if (failed) {
#pragma unroll
        for (int t = 0; t < NT; ++t) { m_run[t] = -INFINITY; l_run[t] = 0.f; }
    }

    // ---- merge the warps in piece space and gather the pieces into channels:
    // c_i = Delta_V o sum_t p_it u_t, still in the transform domain.  A unit with
    // several splits leaves (m, l, c) per query head in its partial slot and the
    // combine kernel applies Uv once per head; a unit with a single split
    // applies Uv here.
    const int rows_tot = 64 * groups;
    float *wm = scr;                                          // [FW][HPG]
    float *wl = wm + FW * HPG;                                // [FW][HPG]
    // [FW][rows_tot][HPG + 1], warp stride wstride: rows padded to an odd number of
    // floats, so that the gather's reads of one head's rows for 32 channels fall in
    // distinct banks (with HPG floats per row they would share HPG-aligned banks)
    constexpr int WROW = HPG + 1;
    float *wacc = reinterpret_cast<float *>(stage_base);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        float l = l_run[t];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (g == 0) {
            wm[warp * HPG + 4 * t + c] = m_run[t];
            wl[warp * HPG + 4 * t + c] = l;
        }
    }
    // the warps' piece sums (unscaled, each against its own running maximum):
    // in the warp's own stages when they hold them (the warp is done with them),
    // else packed over all stages once every warp is out of its loop
    const bool own = (size_t)rows_tot * WROW * 4 <= (size_t)FST * SB;
    const int wstride = own ? (int)(FST * SB / 4) : rows_tot * WROW;   // floats between warps
    if (!own) __syncthreads();
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int i = 4 * t + c;
#pragma unroll
        for (int gr = 0; gr < GMAX; ++gr) {
            if (gr >= groups) break;
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4) {
                const int row = (gr * 4 + m4) * 16 + g;
                wacc[(size_t)warp * wstride + row * WROW + i] = acc[gr][m4][t][0];
                wacc[(size_t)warp * wstride + (row + 8) * WROW + i] = acc[gr][m4][t][1];
            }
        }
    }
    // a wait that gave up in any warp invalidates the whole split
    failed = __syncthreads_or(failed);
    // thread (head i, channel j): merge the warps by log-sum-exp and gather the
    // channel's pieces: c_ij = Delta_V,j sum_w 2^(m_w - M) sum_t p_t u_tj
    // (both sides carry 2^PSH), straight to the partial slot (several splits)
    // or to shared memory (the unit's only split); l likewise
    float *Pg = a.part + ((size_t)u * a.S_slots + sp) * HPG * PROW;
    for (int e = tid; e < HPG * D; e += NTH) {
        const int i = e >> 7, j = e & (D - 1);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < FW; ++w) M = fmaxf(M, wm[w * HPG + i]);
        float f[FW];
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < FW; ++w) {
            const float mw = wm[w * HPG + i];
            f[w] = mw == -INFINITY ? 0.f : ex2(mw - M);
            Ls = fmaf(wl[w * HPG + i], f[w], Ls);
        }
        float v = 0.f;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
            const int vg = blob_s->vgat[j][q2];
            if (vg >= 0) {
                const float *src = wacc + (size_t)(vg & 255) * WROW + i;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int w = 0; w < FW; w += 2) {
                    s0 = fmaf(f[w], src[(size_t)w * wstride], s0);
                    if (w + 1 < FW) s1 = fmaf(f[w + 1], src[(size_t)(w + 1) * wstride], s1);
                }
                // fp16 operands: piece * 2^(p - 24); piece * 2^ex is the code part
                v = fmaf(s0 + s1, pow2i((vg >> 8) - 64 + 24), v);
            }
        }
        v *= blob_s->vstep[j];
        if (a.single) {
            cf[i * D + j] = v;
            if (j == 0) cl[i] = Ls;
            float mx = fabsf(v);   // a warp's 32 channels share one head
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) atomicMax(&mxc[i], __float_as_int(mx));
        } else {
            Pg[i * PROW + 4 + j] = failed ? 0.f : v;
            if (j < 4) Pg[i * PROW + j] = j == 0 ? (failed ? -INFINITY : M) : j == 1 ? (failed ? 0.f : Ls) : 0.f;
        }
    }
    if (!a.single) {
        // count this split in: after the barrier, one thread's atomic add
        // with acquire-release semantics at GPU scope publishes the partial the
        // whole CTA wrote and, for the split counted in last, acquires the
        // others' partials; that split merges the unit and puts the counter
        // back to 0
        __syncthreads();
        if (tid == 0) {
            unsigned old;
            asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.counter + u) : "memory");
            if (old >= (unsigned)a.S_slots) atomicOr(a.status, AATC_DEV_WORKSPACE);   // counters were not zero
            const bool last = old == (unsigned)(a.S_slots - 1);
            if (last) a.counter[u] = 0u;
            mxi[0] = last;
        }
        __syncthreads();
        if (!mxi[0]) {
            mbar_wait(mat_bar, 1);   // (long landed) no copy may be in flight when the CTA exits
            return;
        }
        merge_unit(a.part + (size_t)u * a.S_slots * HPG * PROW, a.S_slots);
    }
    apply_uv(b, h, hg, failed, 1u);
}

// Per-head fast-decoder tables from the plans and codec tables.
__global__ void k_dec_build(const HeadPlan *__restrict__ plans, const CodecTables *__restrict__ tabs, int Wk, int Wv,
                            const double *__restrict__ Ak, const double *__restrict__ Uv, const double *__restrict__ muv,
                            DecBlob *__restrict__ out, float *__restrict__ vcst, uint16_t *__restrict__ dmat)
{
    const int h = blockIdx.x, tid = threadIdx.x;
    const HeadPlan &pk = plans[h * 2 + 0];
    const HeadPlan &pv = plans[h * 2 + 1];
    const CodecTables &tk = tabs[h * 2 + 0];
    const CodecTables &tv = tabs[h * 2 + 1];
    // mu_v - Uv (Delta_V o mid): the part of every output that does not depend on the tokens
    for (int j = tid; j < D; j += blockDim.x) {
        double acc = muv[(size_t)h * D + j];
        for (int k = 0; k < D; ++k)
            if (tv.bits[k]) acc -= Uv[((size_t)h * D + j) * D + k] * ((double)tv.step[k] * (double)tv.mid[k]);
        vcst[(size_t)h * D + j] = (float)acc;
    }
    DecBlob &o = out[h];
    const int rows_tot = 64 * ((2 * Wv + 7) / 8);
    for (int e = tid; e < 16 * 16; e += blockDim.x) {
        const int w = e >> 4, k = e & 15;
        o.kmask[w][k] = w < Wk ? pk.mask[w][k] : 0u;
        for (int half = 0; half < 2; ++half) {
            const int ch = w < Wk ? pk.ch[w][k][half] : -1;
            o.kslot[w][k][half] = (int16_t)(ch < 0 ? -1 : (ch | ((pk.ex[w][k][half] + 64) << 8)));
        }
    }
    for (int e = tid; e < 32 * 8; e += blockDim.x) {
        const int hw = e >> 3, k = e & 7;
        o.vmask[hw][k] = hw < 2 * Wv ? pv.mask[hw][k] : 0u;
    }
    // fp16 operands of the fast decoder's two matrix products, each entry as
    // an fp16 part and the fp16 rounding of what it leaves (about 22
    // significant bits): row j of A_k scaled by 2^(13 - e_j), 2^e_j <= its
    // largest |entry| < 2^(e_j + 1) (the 2^(e_j - 13) goes into ksc_j), and
    // row j of Uv (entries in [-1, 1]) scaled by 2^13.  16-byte chunk n of a
    // row r sits at chunk n ^ (r % 8), so that the eight rows an ldmatrix
    // phase reads fall in distinct shared-memory banks.
    int e_row[(D + 127) / 128];
    for (int j = tid, q = 0; j < D; j += blockDim.x, ++q) {
        const double *ar = Ak + ((size_t)h * D + j) * D;
        const double *ur = Uv + ((size_t)h * D + j) * D;
        double mx = 0.0;
        for (int k = 0; k < D; ++k) mx = fmax(mx, fabs(ar[k]));
        int ex = 0;
        if (mx > 0.0) frexp(mx, &ex);
        const int ej = max(-100, min(100, ex - 1));
        e_row[q] = ej;
        const double sa = ldexp(1.0, 13 - ej);
        uint16_t *Ah = dmat + (size_t)h * 4 * D * D, *Al = Ah + D * D, *Uh = Ah + 2 * D * D, *Ul = Ah + 3 * D * D;
        for (int k = 0; k < D; ++k) {
            const int pos = j * D + ((((k >> 3) ^ (j & 7)) << 3) | (k & 7));
            const double xa = ar[k] * sa, xu = ur[k] * 8192.0;
            const __half ah = __double2half(xa), uh = __double2half(xu);
            const __half al = __double2half(xa - (double)__half2float(ah));
            const __half ul = __double2half(xu - (double)__half2float(uh));
            Ah[pos] = __half_as_ushort(ah);
            Al[pos] = __half_as_ushort(al);
            Uh[pos] = __half_as_ushort(uh);
            Ul[pos] = __half_as_ushort(ul);
        }
    }
    for (int j = tid, q = 0; j < D; j += blockDim.x, ++q) {
        o.ksc[j] = tk.bits[j] ? tk.step[j] * 0.08838834764831845f * pow2i(e_row[q] - 13) : 0.f;
        o.vstep[j] = tv.bits[j] ? tv.step[j] : 0.f;
        // value pieces of channel j: row (gr, m4, rr) holds slot 2 m4 + rr / 8 of half-word 8 gr + rr % 8
        int n = 0;
        int16_t got[2] = {-1, -1};
        for (int row = 0; row < rows_tot && n < 2; ++row) {
            const int gr = row >> 6, m4 = (row >> 4) & 3, rr = row & 15;
            const int hw = 8 * gr + (rr & 7), k = 2 * m4 + (rr >> 3);
            if (hw < 2 * Wv && pv.ch[hw][k][0] == j) got[n++] = (int16_t)(row | ((pv.ex[hw][k][0] + 64) << 8));
        }
        o.vgat[j][0] = got[0];
        o.vgat[j][1] = got[1];
    }
}

template <int GMAX, int NT, int FW>
int occupancy_of(size_t smem)
{
    auto kern = k_decode_fast<GMAX, NT, FW, AATC_PIECES, __nv_bfloat16, false>;   // (the KP = 8 variants use as many registers)
    // through the raise-only helper: setting the attribute directly could lower it
    // below what an earlier launch of this variant, with more shared memory, relies on
    if (kernel_smem_limit((const void *)kern, smem) != AATC_OK) return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, FW * 32, smem) != cudaSuccess || n < 1) n = 1;
    return n;
}

int fast_ctas_per_sm_uncached(int GMAX, int NT, size_t smem)
{
    if (NT == 1) {
        if (GMAX == 2) return occupancy_of<2, 1, 16>(smem);
        if (GMAX == 3) return occupancy_of<3, 1, 16>(smem);
        return occupancy_of<4, 1, 16>(smem);
    }
    if (GMAX == 2) return occupancy_of<2, 2, 12>(smem);
    if (GMAX == 3) return occupancy_of<3, 2, 12>(smem);
    return occupancy_of<4, 2, 12>(smem);
}

int fast_ctas_per_sm(int GMAX, int NT, int FW, size_t smem)
{
    // the answer depends only on the kernel variant and its shared memory
    static struct { int GMAX, NT, FW; size_t smem; int n; } cache[16];
    static int used = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].GMAX == GMAX && cache[i].NT == NT && cache[i].FW == FW && cache[i].smem == smem)
            return cache[i].n;
    const int n = fast_ctas_per_sm_uncached(GMAX, NT, smem);
    if (used < 16) cache[used++] = {GMAX, NT, FW, smem, n};
    return n;
}

// Largest dynamic shared memory of one block on this device.
int sm_limit_bytes()
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
    CacheMap map, const int32_t *__restrict__ seq_lens, int L, int Hkv, int G, int Wk, int Wv, int chunk,
    int n_split, const HeadPlan *__restrict__ plans, const CodecTables *__restrict__ tabs,
    float *__restrict__ part, uint32_t *status)
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

    bool bad_blk = false;
    for (int tok0 = begin; tok0 < end; tok0 += DEC_TILE) {
        const int tok = tok0 + t;
        const bool valid = tok < end;
        uint32_t rec[GEN_MAX_W + 1];
        float sc[AATC_MAX_G];
#pragma unroll
        for (int gg = 0; gg < AATC_MAX_G; ++gg) sc[gg] = -INFINITY;
        if (valid) {
            long long tw = cache_tile_word(map, b, h, Hkv, Wk, tok >> 5);
            long long twv = cache_tile_word(map, b, h, Hkv, Wv, tok >> 5);
            if (tw < 0 || twv < 0) {   // no block for this tile: read tile 0 of the pool, report it
                bad_blk = true;
                tw = twv = 0;
            }
            const uint32_t *tile = kp + tw;
            for (int w = 0; w < Wk; ++w) rec[w] = tile[key_word_pos(tok & 31, w, Wk)];
            rec[Wk] = 0u;
#pragma unroll
            for (int gg = 0; gg < AATC_MAX_G; ++gg) sc[gg] = 0.f;
            for (int j = 0; j < D; ++j) {
                if (!bk[j]) continue;
                const float u = (float)code_at(rec, offk[j], bk[j]);
#pragma unroll
                for (int gg = 0; gg < AATC_MAX_G; ++gg)
                    if (gg < G) sc[gg] = fmaf(q_s[gg][j], u, sc[gg]);
            }
            const uint32_t *vt = vp + twv;
            for (int w = 0; w < Wv; ++w) {
                const uint32_t lo = (vt[16 * (2 * w) + ((tok & 31) >> 1)] >> (16 * (tok & 1))) & 0xFFFFu;
                const uint32_t hi = (vt[16 * (2 * w + 1) + ((tok & 31) >> 1)] >> (16 * (tok & 1))) & 0xFFFFu;
                rec[w] = lo | (hi << 16);
            }
            rec[Wv] = 0u;
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
    if (bad_blk) atomicOr(status, AATC_DEV_RANGE);
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

template <typename K>
aatc_status launch_variant(K kern, int FW, const FastGeom &f, const FastArgs &a, cudaStream_t s)
{
    aatc_status st = kernel_smem_limit((const void *)kern, f.smem);
    if (st != AATC_OK) return st;
    // programmatic dependent launch: the prologue that reads only the handle
    // overlaps the tail of the previous kernel on the stream
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(f.grid);
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

template <int GMAX, int NT, int FW, int KP, int WK = 0, int WV = 0, int FSTC = 0>
aatc_status launch_fast(const FastGeom &f, const FastArgs &a, aatc_dtype dt, cudaStream_t s)
{
    if (a.map.table) {
        if (dt == AATC_BF16)
            return launch_variant(k_decode_fast<GMAX, NT, FW, KP, __nv_bfloat16, true, WK, WV, FSTC>, FW, f, a, s);
        return launch_variant(k_decode_fast<GMAX, NT, FW, KP, float, true, WK, WV, FSTC>, FW, f, a, s);
    }
    if (dt == AATC_BF16)
        return launch_variant(k_decode_fast<GMAX, NT, FW, KP, __nv_bfloat16, false, WK, WV, FSTC>, FW, f, a, s);
    return launch_variant(k_decode_fast<GMAX, NT, FW, KP, float, false, WK, WV, FSTC>, FW, f, a, s);
}

// The kernel with the widths as constants, for the equal K/V widths of 2.0,
// 2.75 and 4.0 bits per element (their pipeline depth as fast_geom picks it);
// false when f is another shape.
template <int NT, int FW>
bool launch_fast_common(const FastGeom &f, const FastArgs &a, aatc_dtype dt, cudaStream_t s, aatc_status *st)
{
    if (f.KP != AATC_PIECES || a.Wk != a.Wv) return false;
    if (a.Wk == 8 && f.FST == 3 && f.GMAX == 2) *st = launch_fast<2, NT, FW, AATC_PIECES, 8, 8, 3>(f, a, dt, s);
    else if (a.Wk == 11 && f.FST == 3 && f.GMAX == 3) *st = launch_fast<3, NT, FW, AATC_PIECES, 11, 11, 3>(f, a, dt, s);
    else if (a.Wk == 16 && f.FST == 2 && f.GMAX == 4) *st = launch_fast<4, NT, FW, AATC_PIECES, 16, 16, 2>(f, a, dt, s);
    else return false;
    return true;
}

// Test hook state (aatc_test_wait_fault): read at every fast-path launch.
std::atomic<int> g_hook_skip{0};
std::atomic<int> g_hook_tries{WAIT_TRIES};


// Arguments of k_decode_fast for geometry f (a plain decode; the fused append
// fills in its fields afterwards).
FastArgs fast_args(const aatc_calib *h, const FastGeom &f, const void *q, const uint32_t *kp, const uint32_t *vp,
                   const CacheMap &map, const int32_t *seq_lens, int L, int B, float *out, void *ws)
{
    FastArgs a;
    a.kp = kp;
    a.vp = vp;
    a.kw = a.vw = nullptr;
    a.seq_lens = seq_lens;
    a.L = L;
    a.map = map;
    a.Wk = h->Wk;
    a.Wv = h->Wv;
    a.rows = f.rows;
    a.groups = f.groups;
    a.Hkv = h->Hkv;
    a.G = h->G;
    a.HG = f.HG;
    a.FST = f.FST;
    a.stage_region = (uint32_t)f.stage_region;
    a.single = f.single ? 1 : 0;
    a.out = out;
    a.vcst = h->vcst;
    a.mats = reinterpret_cast<const __half *>(h->dmat);
    a.n_tiles = f.n_tiles;
    a.units = f.units;
    a.S = f.S > 0 ? f.S : 1;
    a.S_slots = f.S;
    a.n_dec = f.units * f.S;
    a.B = B;
    a.n_new = 0;
    a.L_old = L;
    a.k_new = a.v_new = nullptr;
    a.TT = a.bk = a.bv = nullptr;
    a.app_one_t = 0;
    a.tabs = nullptr;
    a.plans = nullptr;
    a.tiles_per = f.tiles_per;
    a.blob = h->dblob;
    a.q = q;
    a.part = f.single ? nullptr : (float *)((char *)ws + WS_COUNTERS);
    a.counter = f.single ? nullptr : (unsigned *)ws;
    {   // slots per merge chunk: what the stages hold, at most MERGE_LD float4 per thread
        const int fit = (int)(f.stage_region / ((size_t)f.HPG * PROW * 4));
        const int ld = MERGE_LD * 4 * (f.FW * 32) / (f.HPG * PROW);
        a.merge_slots = fit < ld ? fit : ld;
    }
    a.status = h->status;
    a.wait_tries = g_hook_tries.load(std::memory_order_relaxed);
    a.skip_first_copy = g_hook_skip.load(std::memory_order_relaxed);
    return a;
}

aatc_status launch_fast_any(const aatc_calib *h, const FastGeom &f, const FastArgs &a, cudaStream_t s)
{
    aatc_status st;
    if (f.NT == 1 ? launch_fast_common<1, 16>(f, a, h->dtype, s, &st) : launch_fast_common<2, 12>(f, a, h->dtype, s, &st))
        return st;
    if (f.NT == 1 && f.KP == AATC_KEY_PIECES) {
        if (f.GMAX == 2) return launch_fast<2, 1, 16, AATC_KEY_PIECES>(f, a, h->dtype, s);
        if (f.GMAX == 3) return launch_fast<3, 1, 16, AATC_KEY_PIECES>(f, a, h->dtype, s);
        return launch_fast<4, 1, 16, AATC_KEY_PIECES>(f, a, h->dtype, s);
    }
    if (f.NT == 1) {
        if (f.GMAX == 2) return launch_fast<2, 1, 16, AATC_PIECES>(f, a, h->dtype, s);
        if (f.GMAX == 3) return launch_fast<3, 1, 16, AATC_PIECES>(f, a, h->dtype, s);
        return launch_fast<4, 1, 16, AATC_PIECES>(f, a, h->dtype, s);
    }
    if (f.GMAX == 2) return launch_fast<2, 2, 12, AATC_PIECES>(f, a, h->dtype, s);
    if (f.GMAX == 3) return launch_fast<3, 2, 12, AATC_PIECES>(f, a, h->dtype, s);
    return launch_fast<4, 2, 12, AATC_PIECES>(f, a, h->dtype, s);
}

}  // namespace

extern "C" aatc_status aatc_set_fused_step(int mode)
{
    if (mode < 0 || mode > 2) return aatc_fail(AATC_ERR_INVALID_ARG, "fused-step mode %d is not 0, 1 or 2", mode);
    g_fuse_mode.store(mode);
    return AATC_OK;
}

extern "C" int aatc_decode_launches(const aatc_calib *calib)
{
    return !calib ? 0 : fast_ok(calib) ? 1 : 3;
}

extern "C" aatc_status aatc_test_wait_fault(int skip_tile_copy, int wait_tries)
{
    g_hook_skip.store(skip_tile_copy ? 1 : 0);
    g_hook_tries.store(wait_tries > 0 ? wait_tries : WAIT_TRIES);
    return AATC_OK;
}

aatc_status dec_build(aatc_calib *h, cudaStream_t s)
{
    k_dec_build<<<h->Hkv, D, 0, s>>>(h->plan, h->tab, h->Wk, h->Wv, h->A_k, h->U_v, h->mu_v, h->dblob, h->vcst,
                                     h->dmat);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

size_t decode_ws_bytes(const aatc_calib *h, int B, int L)
{
    if (fast_ok(h)) return fast_geom(h, B, L).ws_total;
    return general_ws_bytes(h, B, L);
}

aatc_status decode_run(const aatc_calib *h, const void *q, const uint32_t *kp, const uint32_t *vp,
                       const CacheMap &map, const int32_t *seq_lens, int L, int B, float *out, void *ws,
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
        if (!f.single && f.units > MAX_COUNTED)
            return aatc_fail(AATC_ERR_UNSUPPORTED, "%d units with several splits each", f.units);
        const FastArgs a = fast_args(h, f, q, kp, vp, map, seq_lens, L, B, out, ws);
        return launch_fast_any(h, f, a, s);
    }
    if (h->Wk > GEN_MAX_W || h->Wv > GEN_MAX_W)
        return aatc_fail(AATC_ERR_UNSUPPORTED, "records of %d / %d words", h->Wk, h->Wv);
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
        qp, kp, vp, map, seq_lens, L, h->Hkv, h->G, h->Wk, h->Wv, p.chunk, p.n_split, h->plan, h->tab, part,
        h->status);
    k_decode_combine<<<dim3(B, h->Hq), D, 0, s>>>(part, p.n_split, h->Hq, h->G, h->tab, h->UvT32,
                                                  h->muv32, out);
    AATC_CUDA(cudaGetLastError());
    return AATC_OK;
}

size_t append_decode_ws_bytes(const aatc_calib *h, int B, int L_old, int n_new)
{
    if (fast_ok(h)) {
        const FastGeom f = fast_geom_append(h, B, L_old);
        if (fused_append_fits(h, f, B, n_new)) return f.ws_total;
    }
    return decode_ws_bytes(h, B, L_old + n_new);
}

aatc_status append_decode_run(const aatc_calib *h, const void *k_new, const void *v_new, int n_new, const void *q,
                              uint32_t *kp, uint32_t *vp, const CacheMap &map, int L_old, int B, float *out,
                              void *ws, size_t ws_bytes, cudaStream_t s)
{
    if (B == 0) return AATC_OK;
    if (fast_ok(h)) {
        const FastGeom f = fast_geom_append(h, B, L_old);
        if (fused_append_fits(h, f, B, n_new)) {
            FastArgs a = fast_args(h, f, q, kp, vp, map, nullptr, L_old, B, out, ws);
            a.single = 0;
            a.S_slots = f.S + 1;
            a.kw = kp;
            a.vw = vp;
            a.n_new = n_new;
            a.L_old = L_old;
            a.k_new = k_new;
            a.v_new = v_new;
            a.TT = h->TkvT32;
            a.app_one_t = f.stage_region < APP_TT ? 1 : 0;
            if (!a.part || !a.counter || ws_bytes < f.ws_total)
                return aatc_fail(AATC_ERR_INVALID_ARG, "workspace of %zu bytes required", f.ws_total);
            a.bk = h->bk32;
            a.bv = h->bv32;
            a.tabs = h->tab;
            a.plans = h->plan;
            return launch_fast_any(h, f, a, s);
        }
    }
    // the two steps as separate calls: the append encoder, then decode over all tokens
    aatc_status st = encode_run(h, k_new, v_new, B, n_new, L_old, nullptr, map, kp, vp, s);
    if (st != AATC_OK) return st;
    return decode_run(h, q, kp, vp, map, nullptr, L_old + n_new, B, out, ws, ws_bytes, s);
}

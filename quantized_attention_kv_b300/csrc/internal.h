// internal.h -- private declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "aatc.h"

#define AATC_D 128          // head dimension
#define AATC_MAXB 8         // widest per-channel code
#define AATC_MAX_G 16       // widest GQA group served by one decode block

// Device status bits (the handle's status word, set with atomicOr).
enum : uint32_t {
    AATC_DEV_NONFINITE = 1u,
    AATC_DEV_NO_CONVERGENCE = 2u,
    AATC_DEV_TIMEOUT = 4u,        // a bounded wait inside a kernel gave up
    AATC_DEV_RANGE = 8u,          // a cache position or block table entry out of range (access skipped)
    AATC_DEV_WORKSPACE = 16u,     // a decode workspace's split counters were not zero at entry
};

// Where the 32-token tiles of the cache of one (batch row b, KV head h) live.
// Contiguous cache: (b, h) starts at word (b*H + h)*L_cap*W.  Paged cache:
// logical block n (tiles n*tpb .. n*tpb + tpb - 1, tpb a power of two) of
// row b is physical block table[b*bpr + n] of the pool, and head h of block p
// starts at word (p*H + h)*tpb*32*W.  Either way a tile is 32*W consecutive
// words.
struct CacheMap {
    const int32_t *table;   // device [B][bpr], or NULL for a contiguous cache
    int bpr;                // blocks per table row (paged)
    int tpb_shift;          // tiles per block = 2^tpb_shift (paged)
    int n_blocks;           // blocks in the pool (paged)
    int L_cap;              // tokens per (row, head) (contiguous)
};

inline CacheMap contiguous_map(int L_cap) { return CacheMap{nullptr, 0, 0, 0, L_cap}; }

// Word offset of tile t of (row b, head h) in a cache of H heads and W-word
// records, or -1 when t is outside the cache or the block table names no
// block of the pool for it.
__device__ __forceinline__ long long cache_tile_word(const CacheMap &m, int b, int h, int H, int W, int t)
{
    if (t < 0) return -1;
    if (!m.table) return (long long)t * 32 < m.L_cap ? ((long long)(b * H + h) * m.L_cap + (long long)t * 32) * W : -1;
    const int n = t >> m.tpb_shift;
    if (n >= m.bpr) return -1;
    const int p = m.table[(size_t)b * m.bpr + n];
    if (p < 0 || p >= m.n_blocks) return -1;
    return ((((long long)p * H + h) << m.tpb_shift) + (t & ((1 << m.tpb_shift) - 1))) * 32LL * W;
}

// Per (KV head, tensor) codec tables, fp32/int, derived from bits and steps.
// One struct per (head, tensor); tensor 0 = K, 1 = V.
struct CodecTables {
    float inv_step[AATC_D];   // 1 / Delta_j (correctly rounded), 0 if b_j = 0
    float mid[AATC_D];        // (2^b_j - 1) / 2, 0 if b_j = 0
    float top[AATC_D];        // 2^b_j - 1
    float step[AATC_D];       // Delta_j
    uint8_t bits[AATC_D];     // b_j
};

// Record layout of one (head, tensor), computed on the host from the bits
// (plan.cu).  Codes are stored whole, LSB first, channels in the order of
// the record-order rule; off[j] is the record bit offset of channel j.
//
// For the fast decoder every byte of the record is cut into its pieces (the
// parts of codes lying in it): at most AATC_PIECES of them for values, at
// most KP (4 or AATC_KEY_PIECES) for keys.  A 32-bit word x of a record
// (keys) or a pair word holding the same half-word of two tokens (values) is
// read through 2 KP masks (KP = 4 for values): slot k < KP is x & mask[k]
// (piece k of bytes 0 and 2 of x, or of byte 0 of both half-words), slot
// k >= KP is (x >> 8) & mask[k] (piece k - KP of bytes 1 and 3).  Each masked
// 16-bit half is a piece value times 2^p, p its bit position in its byte, and
// read as an fp16 it equals piece * 2^(p-24) exactly (exponent field 0).
#define AATC_PIECES 4
#define AATC_KEY_PIECES 8         // a byte holds at most 8 pieces (each at least one bit)
#define AATC_PLAN_SLOTS 32    // record words (keys) or half-words (values) covered
struct HeadPlan {
    int16_t off[AATC_D];                  // record bit offset of each code, -1 if pruned
    int16_t order[AATC_D];                // channels in record order (first n_coded entries)
    int32_t n_coded;                      // channels with b_j > 0
    int32_t max_pieces;                   // largest number of pieces in one byte
    uint32_t mask[AATC_PLAN_SLOTS][16];   // keys: per record word; values: per half-word (8 slots)
    int8_t ch[AATC_PLAN_SLOTS][16][2];    // channel of the piece in the low/high half, -1 = none
    int8_t ex[AATC_PLAN_SLOTS][16][2];    // code bit offset of the piece minus p
};

// Per-KV-head tables of the fast decoder, laid out as they sit in shared
// memory (one bulk copy per CTA).  Built on the device from the plans and
// codec tables (decode.cu).
struct __align__(16) DecBlob {
    uint32_t kmask[16][16];    // key record word w, slot k < 2 KP: AND mask (0 past the record)
    uint32_t vmask[32][8];     // value half-word e, slot k: AND mask in both halves
    float ksc[AATC_D];         // Delta_K,j / sqrt(d) times 2^(e_j - 13) (the row scale of the fp16 A_k rows), 0 for pruned channels
    float vstep[AATC_D];       // Delta_V,j, 0 for pruned channels
    int16_t kslot[16][16][2];  // key piece of (word, slot, half): ch | (ex + 64) << 8, -1 = none
    int16_t vgat[AATC_D][2];   // value channel j: its piece rows, row | (ex + 64) << 8, -1 = none
};

// Encoder epilogue constants of one record-order column n (channel order[n]):
// v = c * inv + off is the quantizer input c/Delta + mid with the bias T mu
// folded in; codes are clamp(rint(v), 0, |top|); past n_coded the range is zero
// (no bits, mul = 0).
struct __align__(16) EncCol {
    float inv, off;
    float top;      // largest code; stored negated when the record word ends with this column's code
    uint32_t mul;   // 2^(bit position of the code in its record word)
};
constexpr int ENC_MAX_WORDS = 32;   // record words per tensor at 8 bits per channel
static_assert(ENC_MAX_WORDS * 32 >= AATC_MAXB * AATC_D, "encoder word table too small");

struct aatc_calib {
    int d, Hkv, Hq, G;
    int Bk, Bv;               // record bits per token and head of keys / values
    int Wk, Wv;               // record words (Bk / 32, Bv / 32)
    int Bpair;                // 2 x the requested budget: what a joint allocation splits
    bool joint;               // the K/V split follows the attention-aware token weights
    aatc_dtype dtype;
    void *arena;              // one cudaMalloc backing every device array below
    // fp64 calibration results, [H] leading (exported by aatc_export_calib)
    double *mu_k, *mu_v;                      // [H][d]
    double *T_k, *T_k_inv, *A_k, *T_v, *U_v;  // [H][d][d]
    double *lam_k, *lam_v, *lam_q;            // [H][d]
    int32_t *bits_k, *bits_v;                 // [H][d]
    float *step_k, *step_v;                   // [H][d]
    double *alpha;                            // [H][2] token weights alpha_K, alpha_V (joint allocation)
    int32_t *split;                           // [2] chosen B_K, B_V (joint allocation; device)
    // fp32 operands of the encode / decode kernels
    float *Tk32, *Tv32;       // [H][d][d] transform rows (coefficient i = row i . x)
    float *TkvT32;            // [H][2][d][d] T_k, T_v transposed ([k][i] = row i, column k), fp32
    float *bk32, *bv32;       // [H][d] T mu
    float *AkT32;             // [H][d][d] (Tk^{-T})^T: q'_j = sum_k AkT32[k][j] q_k
    float *UvT32;             // [H][d][d] Uv^T: o_j = sum_k UvT32[k][j] c_k
    float *muv32;             // [H][d]
    CodecTables *tab;         // [H][2]
    HeadPlan *plan;           // [H][2] record layout and decode masks
    DecBlob *dblob;           // [H] fast-decoder tables
    uint16_t *dmat;           // [H][4][d][d] fp16 operands of the fast decoder's matrix products:
                              // A_k rows scaled by powers of two (hi, lo parts), Uv 2^13 (hi, lo);
                              // 16-byte chunk n of row r stored at chunk n ^ (r % 8)
    float *vcst;              // [H][d] mu_v - Uv (Delta_V o mid)
    // tensor-core encoder operands (bf16 inputs): T split in three bf16 terms
    // T = T1 + T2 + T3 with rows in record order, [H][2][3][d][d]; and the
    // epilogue columns [H][2][d]
    void *T3;
    EncCol *enc_cols;
    uint32_t *enc_wfix;       // [H][2][ENC_MAX_WORDS] constant the encoder epilogue subtracts from each record word
    alignas(64) unsigned char tmap_T3[128];   // CUtensorMap over T3 (rows x 128 bf16)
    bool tmap_ok;
    bool fast_layout;         // every value byte holds <= AATC_PIECES pieces (key bytes: at most 8 anyway)
    int kpieces;              // KP: key pieces per byte the fast decoder reads (4, or 8 when a key byte holds more than 4)
    uint32_t *status;         // device status word
};

// ---- error reporting (api.cu) ----
aatc_status aatc_fail(aatc_status st, const char *fmt, ...);
aatc_status aatc_cuda_fail(cudaError_t e, const char *what);
// Raise a kernel's dynamic shared memory limit to `bytes` on the current
// device, with a runtime call only the first time (per device and kernel)
// or for a larger size.
aatc_status kernel_smem_limit(const void *kern, size_t bytes);
#define AATC_CUDA(call)                                                   \
    do {                                                                  \
        cudaError_t _e = (call);                                          \
        if (_e != cudaSuccess) return aatc_cuda_fail(_e, #call);          \
    } while (0)

// ---- calibration kernels (calib.cu) ----
// Runs the whole device calibration pipeline for handle h on stream s.
// Inputs as in aatc_calibrate.  Scratch is taken from `work` (bytes from
// calib_work_bytes).  Returns a launch error, device conditions go to h->status.
size_t calib_work_bytes(int Hkv, int Hq, int N);
aatc_status calib_run(aatc_calib *h, const void *k_cal, const void *v_cal, const void *q_cal,
                      int N, int max_sweeps, void *work, cudaStream_t s);
// Second moments of bf16 rows on the tensor cores (cov_tc.cu):
// S[h] = (1/count) sum_t (x_t - c_h)(x_t - c_h)^T over the `rows` rows of head
// h (X: [H][rows][d]; center [H][d] fp64 or NULL), exact up to one rounding of
// x - c to 28-bit fixed point.  Scratch of cov_tc_scratch(H, rows) bytes.
size_t cov_tc_scratch(int H, long rows);
aatc_status cov_tc_run(const __nv_bfloat16 *X, int H, long rows, const double *center, double *S, long count,
                       void *scratch, uint32_t *status, cudaStream_t s);
// Rebuild the fp32 operands and codec tables from the fp64 results.
aatc_status calib_derive(aatc_calib *h, cudaStream_t s);

// ---- record layout (plan.cu) ----
// Build the plans of every head from host copies of the bits ([H][d] each)
// and upload them to h->plan.  Synchronous.
aatc_status plan_build(aatc_calib *h, const int32_t *bits_k, const int32_t *bits_v);
// Host-side plan of one bit allocation (exposed for the ABI tests).
void plan_one(const int32_t *bits, int W, int kp, HeadPlan *out);

// Build T3, enc_cols and the T3 tensor map (after the plans are on the device).
aatc_status enc_build(aatc_calib *h, cudaStream_t s);
// 2D tensor map (written to 128 bytes at map128, 64-byte aligned) over bf16
// rows of `inner` elements: 64 x 128 boxes, 128-byte swizzle.  False if the
// driver entry point is missing or rejects the layout.
bool tma_map_bf16(void *map128, const void *base, unsigned long long inner, unsigned long long rows);
// Build the fast decoder's per-head tables (after the plans are on the device).
aatc_status dec_build(aatc_calib *h, cudaStream_t s);

// ---- encode (encode.cu, encode_tc.cu) ----
// Token n of row b goes to position (row_start ? row_start[b] : start_pos) + n
// of the cache `map` describes (row_start: device [B], read on the device).
aatc_status encode_tc_run(const aatc_calib *h, const void *k, const void *v, int B, int L_new,
                          int start_pos, const int32_t *row_start, const CacheMap &map, uint32_t *kp,
                          uint32_t *vp, cudaStream_t s);
aatc_status encode_run(const aatc_calib *h, const void *k, const void *v, int B, int L_new,
                       int start_pos, const int32_t *row_start, const CacheMap &map, uint32_t *kp,
                       uint32_t *vp, cudaStream_t s);

// ---- decode (decode.cu) ----
// Host checks of aatc_decode_attention's arguments other than the workspace
// (api.cu); AATC_OK also for B == 0 (nothing to do).
aatc_status decode_check_args(const aatc_calib *calib, const void *q, const uint32_t *k_packed,
                              const uint32_t *v_packed, int L_cap, const int32_t *seq_lens, int L, int B,
                              const float *out);
size_t decode_ws_bytes(const aatc_calib *h, int B, int L);
size_t append_decode_ws_bytes(const aatc_calib *h, int B, int L_old, int n_new);
aatc_status append_decode_run(const aatc_calib *h, const void *k_new, const void *v_new, int n_new, const void *q,
                              uint32_t *kp, uint32_t *vp, const CacheMap &map, int L_old, int B, float *out,
                              void *ws, size_t ws_bytes, cudaStream_t s);
aatc_status decode_run(const aatc_calib *h, const void *q, const uint32_t *kp, const uint32_t *vp,
                       const CacheMap &map, const int32_t *seq_lens, int L, int B, float *out, void *ws,
                       size_t ws_bytes, cudaStream_t s);

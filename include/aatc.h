/*
 * aatc.h -- C ABI of the B300 (sm_103a) library for Attention-Aware Transform
 * Coding (AATC) of LLM KV caches: calibrate a per-head transform and bit
 * allocation, encode keys/values into a fixed-width bit-packed per-token
 * record, and run decode attention directly over the packed cache.
 *
 * Sources of the operations (page title, section):
 *   [ABS]  "KV Cache Compression Through the Lens of Transform Coding", Abstract:
 *          allocate bits over a calibration set to minimize attention-aware
 *          distortion, using transform coding and reverse water-filling.
 *   [KLT]  "Attention-Aware Transform Coding Guide: KV Compression",
 *          "Decorrelation via the Karhunen-Loeve Transform (KLT)".
 *   [RWF]  same page, "Optimal Bit Allocation via Reverse Water-Filling".
 *   [ATT]  same page, "Formal Attention Distortion Model":
 *          o = softmax(q K^T / sqrt(d)) V over the quantized K, V.
 *   [THM]  same page, "Theorem: Additive Error Decomposition" (key error is
 *          weighted by the query, value error by the attention weights).
 *   [IMPL] same page, "End-to-End Implementation" (calibrate, rotate,
 *          quantize per channel).
 *   [SERVE] same page, "Deployment Guide: Integrating AATC with vLLM"
 *          (offline calibration, then a serving engine's decode steps on
 *          the compressed cache).
 *   [NOVA] "Spend Bits Where Queries Look: KV Cache Vector Quantization with
 *          Attention-Preserving Transforms", Abstract: non-orthogonal key
 *          transform (generalized Parseval), fixed per-token bit count,
 *          bandwidth-bound decoding.
 *
 * Conventions for every entry point
 *   - Tensors are caller-owned, contiguous, row-major DEVICE pointers unless
 *     a parameter says "host".  Device pointers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All device work is enqueued on it; only aatc_calibrate and
 *     aatc_check synchronize it.
 *   - Every call returns an aatc_status; no exception crosses the ABI.
 *     Argument errors are found on the host before any launch.  Conditions
 *     only the device can see (non-finite inputs, an eigensolver that did not
 *     converge) set a status word inside the handle, reported by the next
 *     aatc_calibrate / aatc_check.  aatc_last_error() gives a message for
 *     the calling thread's last failure.
 *   - head_dim is 128.  Query head h uses KV head h / G, G = n_q_heads / n_kv_heads.
 *   - Nothing traps, and no kernel waits on another block.
 */
#ifndef AATC_H
#define AATC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    AATC_OK = 0,
    AATC_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size or shape */
    AATC_ERR_UNSUPPORTED = 2,    /* head_dim != 128, budget not a multiple of 32 bits, ... */
    AATC_ERR_CUDA = 3,           /* a CUDA runtime call failed */
    AATC_ERR_NO_CONVERGENCE = 4, /* Jacobi did not converge within jacobi_max_sweeps */
    AATC_ERR_NONFINITE = 5,      /* NaN/Inf in calibration or cache input */
    AATC_ERR_CAPACITY = 6,       /* start_pos + L_new > L_cap, L > L_cap, or a position / block out of range */
    AATC_ERR_TIMEOUT = 7         /* a bounded wait inside a kernel gave up (reported by aatc_check) */
} aatc_status;

typedef enum { AATC_F32 = 0, AATC_BF16 = 1 } aatc_dtype;

/* Opaque calibration handle, owned by the library (aatc_free). */
typedef struct aatc_calib aatc_calib;

typedef struct {
    int head_dim;             /* must be 128 */
    int n_kv_heads;           /* H_kv >= 1 */
    int n_q_heads;            /* H_q, a multiple of H_kv (GQA group G = H_q / H_kv <= 16) */
    int n_calib_tokens;       /* N >= 2 calibration tokens per head */
    double bits_per_element;  /* average bits R; B = 128*R must be an integer multiple
                                 of 32 and at most 8*128 (e.g. 2.0, 2.75, 4.0) */
    aatc_dtype dtype;         /* element type of every K/V/Q input of this handle */
    int jacobi_max_sweeps;    /* <= 0 selects 50 */
    int joint_kv;             /* 0: keys and values get B bits each.  Nonzero: the
                                 pair budget 2B is split between keys and values
                                 (B_K + B_V = 2B, both multiples of 32, each at
                                 most 8*128), one split for every KV head, by the
                                 attention-aware token weights (see aatc_calibrate) */
} aatc_calib_desc;

/* Calibration ([ABS], [KLT], [RWF], [THM], [NOVA]).
 * k_cal, v_cal: device [H_kv][N][128]; q_cal: device [H_q][N][128], all of
 * desc->dtype.  Per KV head it computes the key mean and centered covariance
 * Sk, the value mean and covariance Sv, and the query second moment Sq pooled
 * over the G query heads of the group; then the whitened key transform
 * Tk = Uk^T Sq^{1/2} (Uk the eigenvectors of Sq^{1/2} Sk Sq^{1/2}) and the value
 * KLT Tv = Uv^T, integer bit widths b_j in 0..8 summing to B for each tensor
 * (the B largest gains lam_j 4^-t, ties to the smaller j then t), and steps
 * Delta_j = s_{b_j} sqrt(lam_j) with s_b the MSE-optimal uniform step for a
 * unit Gaussian.  On success *out receives a new handle (free with aatc_free).
 * Precision: fp32 inputs accumulate the moments in fp64.  bf16 inputs compute
 * them on the tensor cores from x - mean rounded once to 28-bit fixed point
 * (one power-of-two scale per channel); the contraction itself is exact, so
 * the moments differ from fp64 ones only by that rounding (relative 2^-27 of
 * each channel's largest |x - mean|).  The eigensolver runs fp32 sweeps,
 * makes their rotations orthogonal in fp64, then runs fp64 sweeps to the fp64
 * stopping test (|a_pq| <= 1e-15 sqrt(|a_pp a_qq|)), so its results are those
 * of an fp64 solver; jacobi_max_sweeps bounds the fp64 sweeps.  Allocation
 * runs in fp64.
 * Synchronizes `stream` once.  Returns NO_CONVERGENCE / NONFINITE from the
 * device status; the handle is not created then. */
aatc_status aatc_calibrate(const aatc_calib_desc *desc, const void *k_cal, const void *v_cal,
                           const void *q_cal, aatc_calib **out, void *stream);

/* Packed cache layout ([NOVA] fixed per-token bit count; the layout itself
 * is this library's reading -- the pages give none).
 *
 * Record: every token of every (KV head, tensor) takes exactly W = B/32
 * little-endian u32 words, record bit k = bit k%32 of word k/32.  The code
 * u_j of each channel with b_j > 0 is stored whole, least significant bit
 * first, in b_j consecutive record bits; pruned channels (b_j = 0) take no
 * bits.  The channels follow one another in this order: start with
 * p2 = p1 = 8; repeatedly take the narrowest remaining channel whose width is
 * at least 7 - p2 - p1 (or the widest remaining one if none is that wide;
 * ties to the lower channel index), then p2 = p1, p1 = its width.
 *
 * Cache: the cache of one (batch row b, KV head h) is L_cap*W words starting
 * at word (b*H_kv + h)*L_cap*W, L_cap a multiple of 32, made of 32-token
 * tiles (tile t = tokens 32t..32t+31, words 32*W*t ..).  Within a tile,
 * token i (0..31):
 *   keys:   record word w is tile word
 *             16*W*(i/16) + 64*r + ((i%16)/2)*2*n_r + 2*(w-4r) + i%2,
 *           r = w/4, n_r = min(4, W-4r);
 *   values: half-word e of the record (bits 16e..16e+15, e < 2W) is bits
 *           16*(i%2)..16*(i%2)+15 of tile word 16*e + i/2.
 * Every cache bit belongs to exactly one record bit. */

/* Encode ([KLT], [IMPL], [NOVA] fixed per-token bit count).
 * k, v: device [B][H_kv][L_new][128] of the handle's dtype, the keys/values of
 * token positions start_pos .. start_pos+L_new-1.  For each row x:
 * c = T (x - mu); u_j = clamp(rint(c_j/Delta_j + (2^b_j - 1)/2), 0, 2^b_j - 1)
 * (round half to even, decided on an fp32 value); the codes are packed into
 * the token's record and placed in the cache as described above.
 * k_packed, v_packed: device u32 caches of B*H_kv*L_cap*W words (layout
 * above); L_cap must be a multiple of 32.  Only the bits of tokens
 * start_pos .. start_pos+L_new-1 are written (value words are shared by two
 * tokens and written 16 bits at a time).  L_new = 0 is a no-op.
 * Kernels: L_new <= 16 (a decode step's new tokens) takes a small append
 * kernel (one CTA per KV head, tensor and row; fp32 transform), launched as a
 * programmatic dependent of the previous kernel on `stream` so that staging T
 * overlaps it; longer bf16 inputs take the tensor-core encoder, fp32 inputs a
 * plain fp32 encoder.
 * Errors: CAPACITY if start_pos + L_new > L_cap; INVALID_ARG if L_cap is not a
 * multiple of 32.  Non-finite inputs set the handle's NONFINITE status (codes
 * of such rows are unspecified). */
aatc_status aatc_encode(const aatc_calib *calib, const void *k, const void *v, int B, int L_new,
                        int start_pos, int L_cap, uint32_t *k_packed, uint32_t *v_packed,
                        void *stream);

/* Decode attention over the packed cache ([ATT], [NOVA] bandwidth-bound decode).
 * q: device [B][H_q][128] of the handle's dtype.  k_packed, v_packed: device
 * caches as written by aatc_encode (L_cap a multiple of 32).  seq_lens: device int32 [B]
 * (tokens 0..seq_lens[b]-1 of row b are attended; each in 0..L) or NULL
 * (every row attends L tokens).  out: device fp32 [B][H_q][128],
 *   out[b][h] = sum_i softmax_i(q . k_hat_i / sqrt(128)) v_hat_i,
 * k_hat/v_hat the decoded keys/values, no causal mask; a row with no tokens
 * gets zeros.  Computed without reconstructing K or V: scores use
 * q' = (Tk^{-T} q) o Delta_K / sqrt(128) against the codes, values are
 * accumulated in the transform domain and the inverse transform Uv is
 * applied once per head.  workspace: device scratch of at least
 * aatc_decode_workspace_size(calib, B, L) bytes, caller-owned; it must hold
 * zeros before its first use (e.g. cudaMemset once when it is allocated),
 * and every call leaves it ready for the next one, whatever the shape; calls
 * that share a workspace must be ordered on one stream.  One kernel is
 * launched on `stream` (as a programmatic dependent of the previous one).
 * When the rows and KV head groups already fill the GPU, each is one CTA
 * that writes `out` directly (no workspace).  Otherwise each (row, KV head
 * group) is split over several CTAs: each leaves a partial result in the
 * workspace -- its running softmax maximum and sum and
 * Delta_V o sum_i p_i u_i over its tokens, in the transform domain -- and
 * counts itself in; the CTA counted in last merges the partials, applies Uv
 * once per query head, adds mu_v - Uv (Delta_V o mid) and writes `out`.
 * Records above 16 words or layouts whose bytes hold more than four code
 * pieces take a slower general path of three kernels.
 * Errors: CAPACITY if L > L_cap; INVALID_ARG if the workspace is too small or
 * L_cap is not a multiple of 32.  A workspace whose counters were not zero
 * at entry sets the handle's status (INVALID_ARG from aatc_check); the
 * output of that call is unspecified. */
aatc_status aatc_decode_attention(const aatc_calib *calib, const void *q,
                                  const uint32_t *k_packed, const uint32_t *v_packed, int L_cap,
                                  const int32_t *seq_lens, int L, int B, float *out,
                                  void *workspace, size_t ws_bytes, void *stream);

/* Bytes of device workspace aatc_decode_attention needs for B rows of up to
 * L tokens.  0 when the call needs none (workspace may then be NULL) and on
 * invalid arguments. */
size_t aatc_decode_workspace_size(const aatc_calib *calib, int B, int L);

/* Decode attention that allocates nothing.  The pages have no counterpart:
 * this is a library convenience.  It computes exactly what
 * aatc_decode_attention computes, with the same arguments except that there
 * is no workspace: the scratch is a fixed 4 MiB array built into the library
 * (every GPU that loads the library holds it until the process exits).  It is
 * meant for callers that cannot hand over device memory -- e.g. an engine
 * plugin whose memory planner has already given out all device memory, or a
 * latency-critical path where cudaMalloc, which may synchronize the device,
 * is not allowed.  It calls no cudaMalloc/cudaFree.
 *   - Shapes needing more scratch than 4 MiB (aatc_decode_workspace_size)
 *     are rejected with AATC_ERR_CAPACITY before any launch.
 *   - Arguments are checked as aatc_decode_attention checks them (same
 *     statuses) before the scratch size is compared with the array.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.  The address is kept for the life of the process: after
 *     a cudaDeviceReset the library must be unloaded and loaded again before
 *     this entry point is used on that device.
 *   - Every call on a device shares the one array.  The first call on a
 *     device also clears the array (cudaMemsetAsync on its stream), which
 *     the split counters need; every call leaves them at zero again.  Calls
 *     that overlap on the GPU -- on different streams, or from several host
 *     threads -- race on it: order them on one stream. */
aatc_status aatc_decode_attention_static(const aatc_calib *calib, const void *q,
                                         const uint32_t *k_packed, const uint32_t *v_packed,
                                         int L_cap, const int32_t *seq_lens, int L, int B,
                                         float *out, void *stream);

/* One decode step of a serving engine in one launch ([SERVE]: the cache
 * grows by each step's new tokens and every step reads it once).  Equivalent to
 *   aatc_encode(calib, k_new, v_new, B, n_new, L_old, L_cap, k_packed, v_packed, stream);
 *   aatc_decode_attention(calib, q, k_packed, v_packed, L_cap, NULL, L_old + n_new, B, out, ...);
 * (the same records written, the same output up to fp32 rounding order),
 * done by one kernel: the decode splits attend the L_old cached tokens while
 * extra CTAs of the same launch encode each (row, KV head)'s n_new tokens
 * (k_new, v_new: device [B][H_kv][n_new][128] of the handle's dtype), write
 * their records at positions L_old .. L_old + n_new - 1, and add the new
 * tokens' attention to the merge as one more partial; no CTA waits for
 * another.  workspace: aatc_append_decode_workspace_size(calib, B, L_old,
 * n_new) bytes, zeroed before its first use (as for aatc_decode_attention;
 * the two may share one workspace).  Shapes the fused kernel does not serve
 * (n_new > 16, records that take the general decode path, more than 256
 * (row, KV head group) pairs) run the two calls above instead.  n_new = 0
 * is aatc_decode_attention over L_old tokens.
 * Errors: as aatc_encode and aatc_decode_attention; CAPACITY if
 * L_old + n_new > L_cap. */
aatc_status aatc_append_decode_attention(const aatc_calib *calib, const void *k_new, const void *v_new, int n_new,
                                         const void *q, uint32_t *k_packed, uint32_t *v_packed, int L_cap,
                                         int L_old, int B, float *out, void *workspace, size_t ws_bytes,
                                         void *stream);

/* Bytes of workspace aatc_append_decode_attention needs (0 on invalid
 * arguments or when it needs none). */
size_t aatc_append_decode_workspace_size(const aatc_calib *calib, int B, int L_old, int n_new);

/* When aatc_append_decode_attention uses its fused kernel (process-wide):
 * 1 (default) when it pays -- the cache is empty, or the decode splits are
 * long enough (48 tiles of 32 tokens per split per (row, KV head) pair an
 * appender CTA takes) that the appenders finish inside them; 2 whenever the
 * shape fits the kernel (for tests); 0 never (append then decode).
 * Workspace sizes follow the mode: size workspaces after setting it.
 * Errors: INVALID_ARG for another mode. */
aatc_status aatc_set_fused_step(int mode);

/* Paged cache ([SERVE]; the layout is this library's).
 * A pool holds n_blocks blocks.  Block p holds block_tokens tokens (32
 * times a power of two: 32, 64, 128, ...) of every KV head: head h of block p is the
 * block_tokens*W words starting at word (p*H_kv + h)*block_tokens*W, tiled
 * exactly as a contiguous cache with L_cap = block_tokens (32-token tiles,
 * layout above).  Logical block n of batch row b (its tokens
 * n*block_tokens .. (n+1)*block_tokens - 1) is physical block
 * block_table[b*blocks_per_row + n].  Rows may share no block they both
 * write.  The table is read on the device, in stream order. */
typedef struct {
    const int32_t *block_table;   /* device [B][blocks_per_row] */
    int blocks_per_row;           /* row stride of block_table, >= 1 */
    int block_tokens;             /* tokens per block: 32 times a power of two */
    int n_blocks;                 /* blocks in each pool, >= 1 */
} aatc_pages;

/* Encode into paged pools (k_pool, v_pool: device u32, n_blocks *
 * H_kv * block_tokens * W words each).  As aatc_encode, except token n of
 * row b goes to logical position row_start[b] + n when row_start (device
 * int32 [B], read on the device) is given, else start_pos + n.  Kernels as
 * aatc_encode; records of a full, 32-aligned tile leave by one bulk store per
 * tile.
 * Errors: INVALID_ARG for a bad `pages` (NULL table, block_tokens not 32
 * times a power of two, ...); CAPACITY if row_start is NULL and
 * start_pos + L_new > blocks_per_row * block_tokens.  A position or block
 * table entry found out of range on the device skips that write and sets the
 * handle's CAPACITY status (reported by aatc_check). */
aatc_status aatc_encode_paged(const aatc_calib *calib, const void *k, const void *v, int B, int L_new,
                              int start_pos, const int32_t *row_start, uint32_t *k_pool, uint32_t *v_pool,
                              const aatc_pages *pages, void *stream);

/* Decode attention over paged pools: as aatc_decode_attention, with the
 * tiles of row b found through the block table (seq_lens / L as there;
 * workspace of aatc_decode_workspace_size(calib, B, L) bytes).  The fast
 * path reads each warp's block table entries three tiles ahead of their
 * copies.
 * Errors: as aatc_decode_attention and aatc_encode_paged; CAPACITY if
 * L > blocks_per_row * block_tokens.  An out-of-range table entry for a tile
 * inside a row's length sets the handle's CAPACITY status (that tile reads
 * block 0). */
aatc_status aatc_decode_attention_paged(const aatc_calib *calib, const void *q, const uint32_t *k_pool,
                                        const uint32_t *v_pool, const aatc_pages *pages, const int32_t *seq_lens,
                                        int L, int B, float *out, void *workspace, size_t ws_bytes, void *stream);

/* Kernels one aatc_decode_attention (or _paged, or _static) call of this
 * handle launches when it has tokens to attend: 1 on the fast path, 3 on the
 * general path (query prep, splits, combine); 0 for a NULL handle.  An
 * aatc_append_decode_attention call launches 1 when its fused kernel serves
 * it. */
int aatc_decode_launches(const aatc_calib *calib);

/* Testing hook (no counterpart in the method): makes a bounded wait inside
 * the decode kernels give up, to exercise the TIMEOUT report without
 * faulting or hanging the GPU.  While skip_tile_copy != 0, every later call
 * of the fast decode path (contiguous or paged) leaves the first tile copy of
 * the first warp of its first CTA unissued; that warp's wait for it gives up
 * after wait_tries tries of at most about 20 us each, the call completes with
 * an unspecified output, and the handle's status reports AATC_ERR_TIMEOUT
 * (aatc_check).  Every copy that was issued is still waited for in full
 * (65,536 tries, about 1.3 s), so nothing is left in flight.
 * aatc_test_wait_fault(0, 0) restores normal operation.  Process-wide; meant
 * for tests only.  Always AATC_OK. */
aatc_status aatc_test_wait_fault(int skip_tile_copy, int wait_tries);

/* W = u32 words per token record of one head (B/32) when keys and values
 * have the same record width, else -1 (see aatc_record_words_kv). */
int aatc_record_words(const aatc_calib *calib);

/* Record words of one tensor: tensor 0 = keys (B_K/32), 1 = values (B_V/32);
 * -1 for a NULL handle or another tensor index.  Key caches hold W_K words
 * per token, value caches W_V; every layout rule above applies with the
 * tensor's own W. */
int aatc_record_words_kv(const aatc_calib *calib, int tensor);

/* Serialize a handle into a caller-owned HOST buffer: a versioned
 * little-endian blob (see aatc_import_calib).  If host_buf is NULL only the
 * size is stored in *bytes; otherwise *bytes must hold the buffer size on
 * entry and receives the bytes written.  Synchronizes the device. */
aatc_status aatc_export_calib(const aatc_calib *calib, void *host_buf, size_t *bytes);

/* Build a handle from a HOST blob.  Layout: int32 header {magic 0x43544141
 * ("AATC"), version 2, head_dim, n_kv_heads, n_q_heads, B_K bits, dtype,
 * B_V bits} (version 1 blobs, whose last word is 0, have B_V = B_K),
 * then for each array below all KV heads in order (H = n_kv_heads, d = 128):
 * f64 mu_k[H][d], mu_v[H][d], T_k[H][d][d], T_k_inv[H][d][d], A_k[H][d][d],
 * T_v[H][d][d], U_v[H][d][d], lam_k[H][d], lam_v[H][d], lam_q[H][d];
 * int32 bits_k[H][d], bits_v[H][d]; f32 step_k[H][d], step_v[H][d].
 * Bits must sum to B_K (keys) and B_V (values) per head, each in 0..8.  Derived device
 * tables (biases, record layout, decode tables) are rebuilt on the device. */
aatc_status aatc_import_calib(const void *host_buf, size_t bytes, aatc_calib **out);

/* Synchronize the device and report (then clear) the handle's device status. */
aatc_status aatc_check(aatc_calib *calib);

/* Release a handle and its device memory.  NULL-safe. */
void aatc_free(aatc_calib *calib);

/* Message describing the calling thread's most recent failure ("" if none). */
const char *aatc_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* AATC_H */

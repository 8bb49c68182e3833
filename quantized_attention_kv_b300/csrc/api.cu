// api.cu -- the C ABI (include/aatc.h): argument checks, handle lifetime,
// calibration blob import/export, status reporting.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <new>

#include "internal.h"

namespace {

thread_local char g_err[512] = "";

constexpr int32_t BLOB_MAGIC = 0x43544141;   // "AATC"
constexpr int32_t BLOB_VERSION = 2;   // version 1 blobs (one budget) still import
constexpr int D = AATC_D;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Sizes of the arena pieces, in the order they are carved.
struct Layout {
    size_t f64_vec, f64_mat, i32_vec, f32_vec, f32_mat, tabs, plans, dblob, dmat, t3, cols, wfix, total;
};

Layout layout_for(int H)
{
    Layout L;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    L.f64_vec = up((size_t)H * D * sizeof(double));
    L.f64_mat = up((size_t)H * D * D * sizeof(double));
    L.i32_vec = up((size_t)H * D * sizeof(int32_t));
    L.f32_vec = up((size_t)H * D * sizeof(float));
    L.f32_mat = up((size_t)H * D * D * sizeof(float));
    L.tabs = up((size_t)H * 2 * sizeof(CodecTables));
    L.plans = up((size_t)H * 2 * sizeof(HeadPlan));
    L.dblob = up((size_t)H * sizeof(DecBlob));
    L.dmat = up((size_t)H * 4 * D * D * 2);
    L.t3 = up((size_t)H * 2 * 3 * D * D * 2);
    L.cols = up((size_t)H * 2 * D * sizeof(EncCol));
    L.wfix = up((size_t)H * 2 * ENC_MAX_WORDS * sizeof(uint32_t));
    L.total = 5 * L.f64_vec + 5 * L.f64_mat + 2 * L.i32_vec + 5 * L.f32_vec + 6 * L.f32_mat + L.tabs +
              L.plans + L.dblob + L.dmat + L.f32_vec + L.t3 + L.cols + L.wfix + 1024 + 2 * L.f64_vec;
    return L;
}

aatc_status new_handle(int Hkv, int Hq, int Bk, int Bv, aatc_dtype dtype, aatc_calib **out)
{
    aatc_calib *h = new (std::nothrow) aatc_calib();
    if (!h) return aatc_fail(AATC_ERR_INVALID_ARG, "out of host memory");
    h->d = D;
    h->Hkv = Hkv;
    h->Hq = Hq;
    h->G = Hq / Hkv;
    h->Bk = Bk;
    h->Bv = Bv;
    h->Wk = Bk / 32;
    h->Wv = Bv / 32;
    h->Bpair = Bk + Bv;
    h->joint = false;
    h->dtype = dtype;
    Layout L = layout_for(Hkv);
    cudaError_t e = cudaMalloc(&h->arena, L.total);
    if (e != cudaSuccess) { delete h; return aatc_cuda_fail(e, "cudaMalloc(handle)"); }
    char *p = (char *)h->arena;
    auto take = [&p](size_t n) { char *r = p; p += n; return r; };
    h->mu_k = (double *)take(L.f64_vec);
    h->mu_v = (double *)take(L.f64_vec);
    h->lam_k = (double *)take(L.f64_vec);
    h->lam_v = (double *)take(L.f64_vec);
    h->lam_q = (double *)take(L.f64_vec);
    h->T_k = (double *)take(L.f64_mat);
    h->T_k_inv = (double *)take(L.f64_mat);
    h->A_k = (double *)take(L.f64_mat);
    h->T_v = (double *)take(L.f64_mat);
    h->U_v = (double *)take(L.f64_mat);
    h->bits_k = (int32_t *)take(L.i32_vec);
    h->bits_v = (int32_t *)take(L.i32_vec);
    h->step_k = (float *)take(L.f32_vec);
    h->step_v = (float *)take(L.f32_vec);
    h->bk32 = (float *)take(L.f32_vec);
    h->bv32 = (float *)take(L.f32_vec);
    h->muv32 = (float *)take(L.f32_vec);
    h->Tk32 = (float *)take(L.f32_mat);
    h->Tv32 = (float *)take(L.f32_mat);
    h->AkT32 = (float *)take(L.f32_mat);
    h->UvT32 = (float *)take(L.f32_mat);
    h->TkvT32 = (float *)take(2 * L.f32_mat);
    h->tab = (CodecTables *)take(L.tabs);
    h->plan = (HeadPlan *)take(L.plans);
    h->dblob = (DecBlob *)take(L.dblob);
    h->dmat = (uint16_t *)take(L.dmat);
    h->vcst = (float *)take(L.f32_vec);
    p = (char *)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);   // T3: TMA source, keep it well aligned
    h->T3 = take(L.t3);
    h->enc_cols = (EncCol *)take(L.cols);
    h->enc_wfix = (uint32_t *)take(L.wfix);
    h->alpha = (double *)take(L.f64_vec);    // [H][2] (fits: H * 128 doubles)
    h->split = (int32_t *)take(256);
    h->status = (uint32_t *)take(256);
    e = cudaMemset(h->status, 0, sizeof(uint32_t));
    if (e != cudaSuccess) { cudaFree(h->arena); delete h; return aatc_cuda_fail(e, "cudaMemset"); }
    *out = h;
    return AATC_OK;
}

aatc_status status_from_device(uint32_t st)
{
    if (st & AATC_DEV_NONFINITE) return aatc_fail(AATC_ERR_NONFINITE, "non-finite value in an input");
    if (st & AATC_DEV_NO_CONVERGENCE)
        return aatc_fail(AATC_ERR_NO_CONVERGENCE, "Jacobi eigensolver did not converge");
    if (st & AATC_DEV_TIMEOUT)
        return aatc_fail(AATC_ERR_TIMEOUT, "a kernel gave up waiting for its own copies; results are invalid");
    if (st & AATC_DEV_WORKSPACE)
        return aatc_fail(AATC_ERR_INVALID_ARG,
                         "a decode workspace was not zeroed before its first use (its split counters were not 0)");
    if (st & AATC_DEV_RANGE)
        return aatc_fail(AATC_ERR_CAPACITY, "a cache position or block table entry was out of range (access skipped)");
    return AATC_OK;
}

aatc_status check_budget(double bits_per_element, int *Bbits)
{
    double b = bits_per_element * D;
    long r = (long)(b + 0.5);
    if (!(bits_per_element > 0.0) || fabs(b - (double)r) > 1e-9 || r % 32 != 0 || r > AATC_MAXB * D)
        return aatc_fail(AATC_ERR_UNSUPPORTED,
                         "bits_per_element=%g: 128*R must be a multiple of 32 in 32..1024", bits_per_element);
    *Bbits = (int)r;
    return AATC_OK;
}

size_t blob_bytes(int H)
{
    const size_t v = (size_t)H * D, m = (size_t)H * D * D;
    return 8 * sizeof(int32_t) + (2 * v + 5 * m + 3 * v) * sizeof(double) + 2 * v * sizeof(int32_t) +
           2 * v * sizeof(float);
}

// Copy the bit allocations back and build the record layouts (one sync).
aatc_status build_plans_from_device(aatc_calib *h)
{
    const size_t n = (size_t)h->Hkv * D;
    int32_t *bk = new (std::nothrow) int32_t[2 * n];
    if (!bk) return aatc_fail(AATC_ERR_INVALID_ARG, "out of host memory");
    cudaError_t e = cudaMemcpy(bk, h->bits_k, n * sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(bk + n, h->bits_v, n * sizeof(int32_t), cudaMemcpyDeviceToHost);
    aatc_status st = e == cudaSuccess ? plan_build(h, bk, bk + n) : aatc_cuda_fail(e, "cudaMemcpy(bits)");
    delete[] bk;
    return st;
}

}  // namespace

aatc_status aatc_fail(aatc_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

aatc_status aatc_cuda_fail(cudaError_t e, const char *what)
{
    return aatc_fail(AATC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

aatc_status kernel_smem_limit(const void *kern, size_t bytes)
{
    // one entry per (device, kernel): the attribute is raised once, and again
    // only for a larger size, so launches on the hot path make no runtime call
    static struct { int dev; const void *k; size_t set; } seen[64];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    AATC_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lock(mu);
    int i = 0;
    while (i < used && !(seen[i].k == kern && seen[i].dev == dev)) ++i;
    if (i < used && seen[i].set >= bytes) return AATC_OK;
    AATC_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
    if (i == used && used < 64) seen[used++] = {dev, kern, 0};
    if (i < used) seen[i].set = bytes;
    return AATC_OK;
}

extern "C" {

const char *aatc_last_error(void) { return g_err; }

aatc_status aatc_calibrate(const aatc_calib_desc *desc, const void *k_cal, const void *v_cal,
                           const void *q_cal, aatc_calib **out, void *stream)
{
    g_err[0] = 0;
    if (!desc || !out) return aatc_fail(AATC_ERR_INVALID_ARG, "desc and out must not be NULL");
    *out = nullptr;
    if (desc->head_dim != D) return aatc_fail(AATC_ERR_UNSUPPORTED, "head_dim must be 128");
    if (desc->n_kv_heads < 1 || desc->n_q_heads < desc->n_kv_heads ||
        desc->n_q_heads % desc->n_kv_heads != 0)
        return aatc_fail(AATC_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
    if (desc->n_q_heads / desc->n_kv_heads > AATC_MAX_G)
        return aatc_fail(AATC_ERR_UNSUPPORTED, "GQA group above 16");
    if (desc->n_calib_tokens < 2) return aatc_fail(AATC_ERR_INVALID_ARG, "need at least 2 calibration tokens");
    if (desc->dtype != AATC_F32 && desc->dtype != AATC_BF16)
        return aatc_fail(AATC_ERR_INVALID_ARG, "unknown dtype");
    if (!k_cal || !v_cal || !q_cal || !aligned16(k_cal) || !aligned16(v_cal) || !aligned16(q_cal))
        return aatc_fail(AATC_ERR_INVALID_ARG, "calibration inputs must be non-NULL and 16-byte aligned");
    int Bbits;
    aatc_status st = check_budget(desc->bits_per_element, &Bbits);
    if (st != AATC_OK) return st;
    const int sweeps = desc->jacobi_max_sweeps > 0 ? desc->jacobi_max_sweeps : 50;
    cudaStream_t s = (cudaStream_t)stream;

    aatc_calib *h = nullptr;
    st = new_handle(desc->n_kv_heads, desc->n_q_heads, Bbits, Bbits, desc->dtype, &h);
    if (st != AATC_OK) return st;
    h->joint = desc->joint_kv != 0;
    void *work = nullptr;
    size_t wb = calib_work_bytes(desc->n_kv_heads, desc->n_q_heads, desc->n_calib_tokens);
    cudaError_t e = cudaMalloc(&work, wb);
    if (e != cudaSuccess) { aatc_free(h); return aatc_cuda_fail(e, "cudaMalloc(calibration scratch)"); }
    st = calib_run(h, k_cal, v_cal, q_cal, desc->n_calib_tokens, sweeps, work, s);
    uint32_t dev = 0;
    if (st == AATC_OK) {
        e = cudaMemcpyAsync(&dev, h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) st = aatc_cuda_fail(e, "calibration");
    } else {
        cudaStreamSynchronize(s);
    }
    if (st == AATC_OK && h->joint) {   // the split chosen on the device sets the record widths
        int32_t sp[2] = {0, 0};
        e = cudaMemcpy(sp, h->split, sizeof(sp), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) st = aatc_cuda_fail(e, "cudaMemcpy(split)");
        h->Bk = sp[0];
        h->Bv = sp[1];
        h->Wk = sp[0] / 32;
        h->Wv = sp[1] / 32;
    }
    cudaFree(work);
    if (st == AATC_OK) st = status_from_device(dev);
    if (st == AATC_OK) st = build_plans_from_device(h);
    if (st != AATC_OK) { aatc_free(h); return st; }
    *out = h;
    return AATC_OK;
}

aatc_status aatc_encode(const aatc_calib *calib, const void *k, const void *v, int B, int L_new,
                        int start_pos, int L_cap, uint32_t *k_packed, uint32_t *v_packed, void *stream)
{
    g_err[0] = 0;
    if (!calib) return aatc_fail(AATC_ERR_INVALID_ARG, "calib is NULL");
    if (B < 0 || L_new < 0 || start_pos < 0 || L_cap < 0)
        return aatc_fail(AATC_ERR_INVALID_ARG, "negative size");
    if (B > 32767 || L_cap > (1 << 28)) return aatc_fail(AATC_ERR_INVALID_ARG, "size too large");
    if (L_cap % 32) return aatc_fail(AATC_ERR_INVALID_ARG, "L_cap = %d is not a multiple of 32", L_cap);
    if ((long)start_pos + L_new > L_cap)
        return aatc_fail(AATC_ERR_CAPACITY, "start_pos + L_new = %ld exceeds L_cap = %d",
                         (long)start_pos + L_new, L_cap);
    if (B == 0 || L_new == 0) return AATC_OK;
    if (!k || !v || !k_packed || !v_packed || !aligned16(k) || !aligned16(v) || !aligned16(k_packed) ||
        !aligned16(v_packed))
        return aatc_fail(AATC_ERR_INVALID_ARG, "tensors must be non-NULL and 16-byte aligned");
    return encode_run(calib, k, v, B, L_new, start_pos, nullptr, contiguous_map(L_cap), k_packed, v_packed,
                      (cudaStream_t)stream);
}

namespace {
aatc_status pages_map(const aatc_pages *pg, CacheMap *m)
{
    if (!pg) return aatc_fail(AATC_ERR_INVALID_ARG, "pages is NULL");
    if (!pg->block_table || ((uintptr_t)pg->block_table & 3u))
        return aatc_fail(AATC_ERR_INVALID_ARG, "block_table must be non-NULL and 4-byte aligned");
    const int tpb = pg->block_tokens / 32;
    if (pg->block_tokens <= 0 || pg->block_tokens % 32 || pg->block_tokens > (1 << 24) || (tpb & (tpb - 1)))
        return aatc_fail(AATC_ERR_INVALID_ARG, "block_tokens = %d is not 32 times a power of two",
                         pg->block_tokens);
    int shift = 0;
    while ((1 << shift) < tpb) ++shift;
    if (pg->blocks_per_row <= 0 || pg->n_blocks <= 0)
        return aatc_fail(AATC_ERR_INVALID_ARG, "blocks_per_row and n_blocks must be positive");
    if ((long long)pg->blocks_per_row * pg->block_tokens > (1LL << 30))
        return aatc_fail(AATC_ERR_INVALID_ARG, "rows of more than 2^30 tokens");
    *m = CacheMap{pg->block_table, pg->blocks_per_row, shift, pg->n_blocks, 0};
    return AATC_OK;
}
}  // namespace

aatc_status aatc_encode_paged(const aatc_calib *calib, const void *k, const void *v, int B, int L_new,
                              int start_pos, const int32_t *row_start, uint32_t *k_pool, uint32_t *v_pool,
                              const aatc_pages *pages, void *stream)
{
    g_err[0] = 0;
    if (!calib) return aatc_fail(AATC_ERR_INVALID_ARG, "calib is NULL");
    if (B < 0 || L_new < 0 || start_pos < 0) return aatc_fail(AATC_ERR_INVALID_ARG, "negative size");
    if (B > 32767) return aatc_fail(AATC_ERR_INVALID_ARG, "size too large");
    CacheMap m;
    aatc_status st = pages_map(pages, &m);
    if (st != AATC_OK) return st;
    const long long row_tokens = (long long)pages->blocks_per_row * pages->block_tokens;
    if (!row_start && (long long)start_pos + L_new > row_tokens)
        return aatc_fail(AATC_ERR_CAPACITY, "start_pos + L_new = %lld exceeds blocks_per_row * block_tokens = %lld",
                         (long long)start_pos + L_new, row_tokens);
    if (row_start && ((uintptr_t)row_start & 3u)) return aatc_fail(AATC_ERR_INVALID_ARG, "row_start misaligned");
    if (B == 0 || L_new == 0) return AATC_OK;
    if (!k || !v || !k_pool || !v_pool || !aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
        return aatc_fail(AATC_ERR_INVALID_ARG, "tensors must be non-NULL and 16-byte aligned");
    return encode_run(calib, k, v, B, L_new, start_pos, row_start, m, k_pool, v_pool, (cudaStream_t)stream);
}

size_t aatc_decode_workspace_size(const aatc_calib *calib, int B, int L)
{
    if (!calib || B < 0 || L < 0) return 0;
    return decode_ws_bytes(calib, B, L);
}

}  // extern "C"

aatc_status decode_check_args(const aatc_calib *calib, const void *q, const uint32_t *k_packed,
                              const uint32_t *v_packed, int L_cap, const int32_t *seq_lens, int L, int B,
                              const float *out)
{
    if (!calib) return aatc_fail(AATC_ERR_INVALID_ARG, "calib is NULL");
    if (B < 0 || L < 0 || L_cap < 0) return aatc_fail(AATC_ERR_INVALID_ARG, "negative size");
    if (B > 65535 || L_cap > (1 << 28)) return aatc_fail(AATC_ERR_INVALID_ARG, "size too large");
    if (L_cap % 32) return aatc_fail(AATC_ERR_INVALID_ARG, "L_cap = %d is not a multiple of 32", L_cap);
    if (L > L_cap) return aatc_fail(AATC_ERR_CAPACITY, "L = %d exceeds L_cap = %d", L, L_cap);
    if (B == 0) return AATC_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out))
        return aatc_fail(AATC_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
    if (L_cap > 0 && (!k_packed || !v_packed || !aligned16(k_packed) || !aligned16(v_packed)))
        return aatc_fail(AATC_ERR_INVALID_ARG, "packed caches must be non-NULL and 16-byte aligned");
    if (seq_lens && ((uintptr_t)seq_lens & 3u)) return aatc_fail(AATC_ERR_INVALID_ARG, "seq_lens misaligned");
    return AATC_OK;
}

extern "C" {

aatc_status aatc_decode_attention(const aatc_calib *calib, const void *q, const uint32_t *k_packed,
                                  const uint32_t *v_packed, int L_cap, const int32_t *seq_lens, int L,
                                  int B, float *out, void *workspace, size_t ws_bytes, void *stream)
{
    g_err[0] = 0;
    aatc_status st = decode_check_args(calib, q, k_packed, v_packed, L_cap, seq_lens, L, B, out);
    if (st != AATC_OK || B == 0) return st;
    const size_t need = decode_ws_bytes(calib, B, L);
    if (need > 0 && (!workspace || !aligned16(workspace) || ws_bytes < need))
        return aatc_fail(AATC_ERR_INVALID_ARG, "workspace of %zu bytes (16-byte aligned) required", need);
    return decode_run(calib, q, k_packed, v_packed, contiguous_map(L_cap), seq_lens, L, B, out, workspace,
                      ws_bytes, (cudaStream_t)stream);
}

aatc_status aatc_append_decode_attention(const aatc_calib *calib, const void *k_new, const void *v_new, int n_new,
                                         const void *q, uint32_t *k_packed, uint32_t *v_packed, int L_cap,
                                         int L_old, int B, float *out, void *workspace, size_t ws_bytes,
                                         void *stream)
{
    g_err[0] = 0;
    if (!calib) return aatc_fail(AATC_ERR_INVALID_ARG, "calib is NULL");
    if (n_new < 0 || L_old < 0) return aatc_fail(AATC_ERR_INVALID_ARG, "negative size");
    if (B > 32767 || n_new > (1 << 28) || L_old > (1 << 28)) return aatc_fail(AATC_ERR_INVALID_ARG, "size too large");
    const int L = L_old + n_new;
    aatc_status st = decode_check_args(calib, q, k_packed, v_packed, L_cap, nullptr, L, B, out);
    if (st != AATC_OK || B == 0) return st;
    if (n_new > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
        return aatc_fail(AATC_ERR_INVALID_ARG, "k_new and v_new must be non-NULL and 16-byte aligned");
    const size_t need = n_new > 0 ? append_decode_ws_bytes(calib, B, L_old, n_new) : decode_ws_bytes(calib, B, L);
    if (need > 0 && (!workspace || !aligned16(workspace) || ws_bytes < need))
        return aatc_fail(AATC_ERR_INVALID_ARG, "workspace of %zu bytes (16-byte aligned) required", need);
    if (n_new == 0)
        return decode_run(calib, q, k_packed, v_packed, contiguous_map(L_cap), nullptr, L, B, out, workspace,
                          ws_bytes, (cudaStream_t)stream);
    return append_decode_run(calib, k_new, v_new, n_new, q, k_packed, v_packed, contiguous_map(L_cap), L_old, B,
                             out, workspace, ws_bytes, (cudaStream_t)stream);
}

size_t aatc_append_decode_workspace_size(const aatc_calib *calib, int B, int L_old, int n_new)
{
    if (!calib || B < 0 || L_old < 0 || n_new < 0 || L_old > (1 << 28) || n_new > (1 << 28)) return 0;
    return n_new > 0 ? append_decode_ws_bytes(calib, B, L_old, n_new) : decode_ws_bytes(calib, B, L_old);
}

aatc_status aatc_decode_attention_paged(const aatc_calib *calib, const void *q, const uint32_t *k_pool,
                                        const uint32_t *v_pool, const aatc_pages *pages, const int32_t *seq_lens,
                                        int L, int B, float *out, void *workspace, size_t ws_bytes, void *stream)
{
    g_err[0] = 0;
    if (!calib) return aatc_fail(AATC_ERR_INVALID_ARG, "calib is NULL");
    if (B < 0 || L < 0) return aatc_fail(AATC_ERR_INVALID_ARG, "negative size");
    if (B > 65535) return aatc_fail(AATC_ERR_INVALID_ARG, "size too large");
    CacheMap m;
    aatc_status st = pages_map(pages, &m);
    if (st != AATC_OK) return st;
    const long long row_tokens = (long long)pages->blocks_per_row * pages->block_tokens;
    if (L > row_tokens)
        return aatc_fail(AATC_ERR_CAPACITY, "L = %d exceeds blocks_per_row * block_tokens = %lld", L, row_tokens);
    if (B == 0) return AATC_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out))
        return aatc_fail(AATC_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
    if (!k_pool || !v_pool || !aligned16(k_pool) || !aligned16(v_pool))
        return aatc_fail(AATC_ERR_INVALID_ARG, "pools must be non-NULL and 16-byte aligned");
    if (seq_lens && ((uintptr_t)seq_lens & 3u)) return aatc_fail(AATC_ERR_INVALID_ARG, "seq_lens misaligned");
    const size_t need = decode_ws_bytes(calib, B, L);
    if (need > 0 && (!workspace || !aligned16(workspace) || ws_bytes < need))
        return aatc_fail(AATC_ERR_INVALID_ARG, "workspace of %zu bytes (16-byte aligned) required", need);
    return decode_run(calib, q, k_pool, v_pool, m, seq_lens, L, B, out, workspace, ws_bytes, (cudaStream_t)stream);
}

int aatc_record_words(const aatc_calib *calib) { return calib && calib->Wk == calib->Wv ? calib->Wk : -1; }

int aatc_record_words_kv(const aatc_calib *calib, int tensor)
{
    if (!calib || (tensor != 0 && tensor != 1)) return -1;
    return tensor ? calib->Wv : calib->Wk;
}

aatc_status aatc_export_calib(const aatc_calib *calib, void *host_buf, size_t *bytes)
{
    g_err[0] = 0;
    if (!calib || !bytes) return aatc_fail(AATC_ERR_INVALID_ARG, "calib and bytes must not be NULL");
    const int H = calib->Hkv;
    const size_t need = blob_bytes(H);
    if (!host_buf) { *bytes = need; return AATC_OK; }
    if (*bytes < need) return aatc_fail(AATC_ERR_INVALID_ARG, "buffer of %zu bytes required", need);
    AATC_CUDA(cudaDeviceSynchronize());
    int32_t hdr[8] = {BLOB_MAGIC, BLOB_VERSION, D, calib->Hkv, calib->Hq, calib->Bk, (int32_t)calib->dtype, calib->Bv};
    char *p = (char *)host_buf;
    memcpy(p, hdr, sizeof(hdr));
    p += sizeof(hdr);
    const size_t v = (size_t)H * D, m = (size_t)H * D * D;
    const void *srcs[] = {calib->mu_k, calib->mu_v, calib->T_k, calib->T_k_inv, calib->A_k, calib->T_v,
                          calib->U_v, calib->lam_k, calib->lam_v, calib->lam_q, calib->bits_k,
                          calib->bits_v, calib->step_k, calib->step_v};
    const size_t sz[] = {v * 8, v * 8, m * 8, m * 8, m * 8, m * 8, m * 8, v * 8, v * 8, v * 8,
                         v * 4, v * 4, v * 4, v * 4};
    for (int i = 0; i < 14; ++i) {
        AATC_CUDA(cudaMemcpy(p, srcs[i], sz[i], cudaMemcpyDeviceToHost));
        p += sz[i];
    }
    *bytes = need;
    return AATC_OK;
}

aatc_status aatc_import_calib(const void *host_buf, size_t bytes, aatc_calib **out)
{
    g_err[0] = 0;
    if (!host_buf || !out) return aatc_fail(AATC_ERR_INVALID_ARG, "host_buf and out must not be NULL");
    *out = nullptr;
    if (bytes < 8 * sizeof(int32_t)) return aatc_fail(AATC_ERR_INVALID_ARG, "blob too short");
    int32_t hdr[8];
    memcpy(hdr, host_buf, sizeof(hdr));
    if (hdr[0] != BLOB_MAGIC || (hdr[1] != 1 && hdr[1] != BLOB_VERSION))
        return aatc_fail(AATC_ERR_INVALID_ARG, "not an AATC calibration blob (version 1 or 2)");
    if (hdr[2] != D) return aatc_fail(AATC_ERR_UNSUPPORTED, "head_dim must be 128");
    const int H = hdr[3], Hq = hdr[4], Bk = hdr[5], Bv = hdr[1] == 1 ? hdr[5] : hdr[7];
    if (H < 1 || Hq < H || Hq % H || Hq / H > AATC_MAX_G)
        return aatc_fail(AATC_ERR_INVALID_ARG, "bad head counts in blob");
    if (Bk <= 0 || Bk % 32 || Bk > AATC_MAXB * D || Bv <= 0 || Bv % 32 || Bv > AATC_MAXB * D)
        return aatc_fail(AATC_ERR_UNSUPPORTED, "bad bit budget in blob");
    if (hdr[6] != AATC_F32 && hdr[6] != AATC_BF16) return aatc_fail(AATC_ERR_INVALID_ARG, "bad dtype");
    if (bytes < blob_bytes(H)) return aatc_fail(AATC_ERR_INVALID_ARG, "blob truncated");
    const size_t v = (size_t)H * D, m = (size_t)H * D * D;
    const char *p = (const char *)host_buf + sizeof(hdr);
    const int32_t *bk = (const int32_t *)(p + (5 * v + 5 * m) * 8);
    const int32_t *bv = bk + v;
    for (int hh = 0; hh < H; ++hh) {
        int sk = 0, sv = 0;
        for (int j = 0; j < D; ++j) {
            int a = bk[hh * D + j], b = bv[hh * D + j];
            if (a < 0 || a > AATC_MAXB || b < 0 || b > AATC_MAXB)
                return aatc_fail(AATC_ERR_INVALID_ARG, "bit width outside 0..8");
            sk += a;
            sv += b;
        }
        if (sk != Bk || sv != Bv) return aatc_fail(AATC_ERR_INVALID_ARG, "bits do not sum to the budget");
    }
    aatc_calib *h = nullptr;
    aatc_status st = new_handle(H, Hq, Bk, Bv, (aatc_dtype)hdr[6], &h);
    if (st != AATC_OK) return st;
    void *dsts[] = {h->mu_k, h->mu_v, h->T_k, h->T_k_inv, h->A_k, h->T_v, h->U_v, h->lam_k, h->lam_v,
                    h->lam_q, h->bits_k, h->bits_v, h->step_k, h->step_v};
    const size_t sz[] = {v * 8, v * 8, m * 8, m * 8, m * 8, m * 8, m * 8, v * 8, v * 8, v * 8,
                         v * 4, v * 4, v * 4, v * 4};
    for (int i = 0; i < 14; ++i) {
        cudaError_t e = cudaMemcpy(dsts[i], p, sz[i], cudaMemcpyHostToDevice);
        if (e != cudaSuccess) { aatc_free(h); return aatc_cuda_fail(e, "cudaMemcpy(import)"); }
        p += sz[i];
    }
    st = calib_derive(h, 0);
    if (st == AATC_OK) st = plan_build(h, bk, bv);
    if (st == AATC_OK) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) st = aatc_cuda_fail(e, "import");
    }
    if (st != AATC_OK) { aatc_free(h); return st; }
    *out = h;
    return AATC_OK;
}

aatc_status aatc_check(aatc_calib *calib)
{
    g_err[0] = 0;
    if (!calib) return aatc_fail(AATC_ERR_INVALID_ARG, "calib is NULL");
    uint32_t dev = 0;
    AATC_CUDA(cudaDeviceSynchronize());
    AATC_CUDA(cudaMemcpy(&dev, calib->status, sizeof(uint32_t), cudaMemcpyDeviceToHost));
    AATC_CUDA(cudaMemset(calib->status, 0, sizeof(uint32_t)));
    return status_from_device(dev);
}

void aatc_free(aatc_calib *calib)
{
    if (!calib) return;
    if (calib->arena) cudaFree(calib->arena);
    delete calib;
}

}  // extern "C"

// decode_static.cu -- decode attention for callers that cannot allocate.
//
// aatc_decode_attention takes its scratch from the caller.  Some callers
// cannot provide one: a plugin inside an inference engine whose memory
// planner has already handed out all device memory, or code on a
// latency-critical path where cudaMalloc (which may synchronize the device)
// is not allowed.  This entry point gives them the same computation with the
// scratch held by the library itself, in a fixed array compiled into this
// file.  It allocates nothing: no cudaMalloc, no cudaFree.
#include <mutex>

#include "internal.h"

// Scratch used by every call on a device.  It lives as long as the library
// is loaded on that device (every GPU that loads the library holds it).
#define AATC_STATIC_SCRATCH_BYTES (4u << 20)   // 4 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[AATC_STATIC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 128;
void *g_scratch_addr[MAX_DEVICES];   // device address of g_decode_scratch, per device
std::mutex g_scratch_mu;

// In host code g_decode_scratch names a host-side stand-in, not device
// memory, so its device address is looked up once per device (with that
// device current) and cached.  At that set-up the array is also cleared on
// the caller's stream: the decode's split counters must start at zero (each
// call leaves them at zero again).
aatc_status scratch_for_current_device(void **out, cudaStream_t s)
{
    int dev = -1;
    AATC_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= MAX_DEVICES) return aatc_fail(AATC_ERR_UNSUPPORTED, "device index %d too large", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return aatc_cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
        e = cudaMemsetAsync(p, 0, AATC_STATIC_SCRATCH_BYTES, s);
        if (e != cudaSuccess) return aatc_cuda_fail(e, "cudaMemsetAsync(decode scratch)");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return AATC_OK;
}

}  // namespace

extern "C" aatc_status aatc_decode_attention_static(const aatc_calib *calib, const void *q,
                                                    const uint32_t *k_packed, const uint32_t *v_packed,
                                                    int L_cap, const int32_t *seq_lens, int L, int B,
                                                    float *out, void *stream)
{
    // the same argument checks as aatc_decode_attention, before the scratch
    // size is worked out from B and L
    aatc_status st = decode_check_args(calib, q, k_packed, v_packed, L_cap, seq_lens, L, B, out);
    if (st != AATC_OK || B == 0) return st;
    const size_t need = decode_ws_bytes(calib, B, L);
    if (need > AATC_STATIC_SCRATCH_BYTES)
        return aatc_fail(AATC_ERR_CAPACITY,
                         "this shape needs %zu bytes of scratch; the built-in scratch holds %u bytes "
                         "(use aatc_decode_attention with a caller workspace)",
                         need, (unsigned)AATC_STATIC_SCRATCH_BYTES);
    void *scratch = nullptr;
    st = scratch_for_current_device(&scratch, (cudaStream_t)stream);
    if (st != AATC_OK) return st;
    // The decode kernels overwrite every other scratch byte before they read
    // it, so nothing else needs clearing between calls.
    return aatc_decode_attention(calib, q, k_packed, v_packed, L_cap, seq_lens, L, B, out, scratch,
                                 AATC_STATIC_SCRATCH_BYTES, stream);
}

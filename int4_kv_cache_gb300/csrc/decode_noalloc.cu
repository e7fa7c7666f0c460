// decode_noalloc.cu -- fused int4 decode for callers that cannot allocate.
//
// tq_sdpa_int4_decode needs a caller-provided workspace for the split-K
// partial states.  Some callers have no way to provide one: code that runs
// where allocation is forbidden or unavailable (inside a host callback, a
// real-time or signal-safe path, a plugin of a framework that owns all device
// memory, or a C program that links only this library and never calls
// cudaMalloc).  This entry point keeps the partial states in a fixed device
// array that belongs to the library instead, so a call allocates nothing.
//
// The array lives in device memory of every GPU that loads the library, for
// as long as the process runs.  All calls on a device share it, and it keeps
// whatever the previous call left: every element a call reads has first been
// written by that same call, so nothing needs clearing, but two calls that can
// run at the same time on the GPU (different streams, or another host thread)
// race on it and may return wrong results.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tq.h"
#include "tq_internal.h"

namespace {

// File-scope scratch: the fp32 partial states (m, l, acc) of one decode call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TQ_NOALLOC_SCRATCH_BYTES];

// The unique id of the calling thread's current context (0 if unknown).  A
// device reset ends the context the array's address was looked up in; the
// next call then sees another id and looks the address up again.
unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static std::once_flag once;
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory; the device address is looked up once per device (and again after a
// reset gave the device a new context) with that device current, and that
// address is what the kernels receive.
tq_status scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    static unsigned long long ctx_of[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tq::record_cuda_status(e);
    if (dev < 0 || dev >= 64) return TQ_ERR_UNSUPPORTED;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the primary context current if none is
        if (e != cudaSuccess || p == nullptr) return tq::record_cuda_status(e != cudaSuccess ? e : cudaErrorUnknown);
        addr[dev] = p;
        ctx_of[dev] = current_context_id();
    }
    *out = addr[dev];
    return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_sdpa_int4_decode_noalloc(const tq_kv_cache* cache, const uint16_t* q,
                                                 int32_t num_q_heads, const int32_t* seq_lens,
                                                 int32_t max_seq_len, float attn_scale, int32_t chunk,
                                                 uint16_t* out, int32_t* status, void* stream) {
    void* scratch = nullptr;
    tq_status s = scratch_address(&scratch);
    if (s != TQ_OK) return s;
    return tq::decode_into_partials(cache, q, num_q_heads, seq_lens, max_seq_len, attn_scale, chunk,
                                    static_cast<uint8_t*>(scratch), TQ_NOALLOC_SCRATCH_BYTES, out, status,
                                    static_cast<cudaStream_t>(stream));
}

// kda_fwd_noalloc: the prefill entry point for callers that cannot allocate
// device memory.
//
// kda_fwd needs a small workspace from its caller (a status word and the
// longest-first launch order of the sequences).  Some callers cannot provide
// one: code that runs where allocation is not allowed or not possible, such as
// a host callback on a stream, a plugin living inside a runtime that owns every
// device allocation, or an embedding with no allocator at all.  For them this
// entry point keeps the scratch in a fixed array inside the library's own
// device memory, so the caller passes only the inputs and outputs.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  Each call starts by clearing the status word (the set-up
// kernel does it) and rewrites the launch order it needs, so nothing carries
// over between calls that run one after another.  Calls that overlap on the
// GPU (for example on two streams at once) share the array and race; issue
// them one after another.
#include <cuda.h>
#include <stdint.h>

#include <mutex>

#include "kda_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes =
    kda::kWsOrderOffset + 4 * static_cast<size_t>(KDA_NOALLOC_MAX_SEQS);

// 65,552 bytes of scratch per GPU that loads the library, held until the
// process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];  // context id the address belongs to

using PfnCtxGetCurrent = CUresult (*)(CUcontext *);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_entry(const char *name) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(f);
}

// Unique id of the context current on this thread (ids are never reused), or
// 0 when it cannot be read.
unsigned long long current_context_id() {
    static const PfnCtxGetCurrent get_current = driver_entry<PfnCtxGetCurrent>("cuCtxGetCurrent");
    static const PfnCtxGetId get_id = driver_entry<PfnCtxGetId>("cuCtxGetId");
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress at set-up -- once per device, with that device current
// -- and cached together with the id of the device's context.  Destroying
// that context (cudaDeviceReset) unloads the library's device code; the next
// call sees a new context id and looks the address up again instead of using
// the stale one.  When the id cannot be read the lookup runs on every call.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    const unsigned long long ctx = current_context_id();
    if (g_scratch_addr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
        // the lookup initialises the context if no call has yet: read the id again
        g_scratch_ctx[dev] = ctx ? ctx : current_context_id();
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status_t kda_fwd_noalloc(const void *q, const void *k, const void *v,
                                        const float *log_alpha, const float *beta,
                                        const float *S0, const int32_t *cu_seqlens, int B,
                                        int T, int H, int d_k, int d_v, int N,
                                        kda_dtype_t dtype, void *o, float *S_T,
                                        int32_t *device_status, void *stream) {
    if (N < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (N > KDA_NOALLOC_MAX_SEQS) return KDA_ERR_WORKSPACE;  // the fixed scratch is too small
    if (device_status && ((uintptr_t)device_status & 3u) != 0) return KDA_ERR_INVALID_ARGUMENT;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    const kda_status_t st =
        kda_fwd_engine(q, k, v, log_alpha, beta, S0, cu_seqlens, B, T, H, d_k, d_v, N, dtype, o,
                       S_T, scratch, kNoAllocScratchBytes, stream, KDA_ENGINE_AUTO);
    if (st != KDA_OK) return st;
    if (device_status &&
        cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

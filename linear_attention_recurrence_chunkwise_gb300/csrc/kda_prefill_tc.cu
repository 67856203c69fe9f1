// Tensor-core (tcgen05 / TMEM / TMA) chunkwise KDA forward for sm_103a.
// Not enabled yet: the engine reports itself unsupported, so kda_fwd routes
// every call to the CUDA-core engine.
#include "kda_internal.h"

namespace kda {

bool prefill_tc_supported(kda_dtype_t, int, int) { return false; }

cudaError_t launch_prefill_tc(const FwdParams &, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace kda

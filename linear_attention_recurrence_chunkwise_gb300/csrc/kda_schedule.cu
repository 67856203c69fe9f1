// Per-call set-up kernel for kda_fwd: clears the workspace status word,
// checks the device-side cu_seqlens, and writes a longest-first launch order
// so that the blocks carrying the longest serial chunk chains start first.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kMaxSortN = 8192;  // above this the order stays the identity

__global__ void __launch_bounds__(1024) schedule_kernel(const int32_t *__restrict__ cu,
                                                         int N, int64_t Ttot,
                                                         int32_t *status, int32_t *order) {
    __shared__ int bad;
    if (threadIdx.x == 0) {
        bad = 0;
        *status = KDA_OK;
    }
    __syncthreads();
    if (!cu) return;
    for (int i = threadIdx.x; i <= N; i += blockDim.x) {
        const int32_t c = cu[i];
        const bool wrong = (i == 0 && c != 0) || (i == N && (int64_t)c != Ttot) ||
                           (i < N && cu[i + 1] < c);
        if (wrong) atomicExch(&bad, 1);
    }
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) *status = KDA_ERR_INVALID_ARGUMENT;
        return;
    }
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        int rank = i;
        if (N <= kMaxSortN) {
            const int li = cu[i + 1] - cu[i];
            rank = 0;
            for (int j = 0; j < N; ++j) {
                const int lj = cu[j + 1] - cu[j];
                rank += (lj > li) || (lj == li && j < i);
            }
        }
        order[rank] = i;
    }
}

}  // namespace

cudaError_t launch_schedule(const FwdParams &p, cudaStream_t s) {
    schedule_kernel<<<1, 1024, 0, s>>>(p.cu_seqlens, p.N, p.Ttot, p.status,
                                       const_cast<int32_t *>(p.order));
    return cudaGetLastError();
}

}  // namespace kda

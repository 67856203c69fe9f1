// Internal declarations shared by the libkda translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;           // tokens per chunk
constexpr float kLogDecayLimit = 80.f;  // |in-chunk cumulative log-decay| supported

// Workspace layout (bytes): [0, 4) int32 status word, [16, 16 + 4N) int32
// launch order of the sequences (longest first).
constexpr size_t kWsOrderOffset = 16;

struct FwdParams {
    const void *q, *k, *v;
    const float *log_alpha, *beta, *S0;
    const int32_t *cu_seqlens;  // nullptr: fixed length T per sequence
    void *o;
    float *S_T;
    int32_t *status;            // workspace status word
    const int32_t *order;       // workspace launch order, nullptr for fixed length
    int64_t Ttot;
    int T;                      // tokens per sequence when cu_seqlens is null
    int H, N, dk, dv;
};

// Token range of sequence n (device helper used by every prefill kernel).
__device__ __forceinline__ void seq_range(const FwdParams &p, int n, int64_t &start,
                                          int &len) {
    if (p.cu_seqlens) {
        start = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - p.cu_seqlens[n];
    } else {
        start = (int64_t)n * p.T;
        len = p.T;
    }
}

__device__ __forceinline__ void raise_status(int32_t *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// The bounds-checked build (KDA_BOUNDS_CHECK=1, the stand-in for a memory
// sanitizer) checks each computed global index against its tensor's extent
// before the access; a failure records KDA_ERR_BOUNDS and the access is
// skipped.  In the normal build the check compiles away.
#ifndef KDA_BOUNDS_CHECK
#define KDA_BOUNDS_CHECK 0
#endif
__device__ __forceinline__ bool in_bounds(int32_t *status, size_t idx, size_t n) {
#if KDA_BOUNDS_CHECK
    if (idx < n) return true;
    raise_status(status, KDA_ERR_BOUNDS);
    return false;
#else
    (void)status, (void)idx, (void)n;
    return true;
#endif
}

cudaError_t launch_schedule(const FwdParams &p, cudaStream_t s);
cudaError_t launch_prefill_simt(const FwdParams &p, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_prefill_tc(const FwdParams &p, cudaStream_t s);
bool prefill_tc_supported(kda_dtype_t dt, int dk, int dv);
cudaError_t launch_verify(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, const float *S, int N, int K, int H, int d,
                          kda_dtype_t dt, void *o, cudaStream_t s);
cudaError_t launch_commit(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, float *S, const int32_t *n_accept, int N, int K,
                          int H, int d, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *log_alpha, const float *beta, float *S, int N,
                          int H, int d, kda_dtype_t dt, void *o, cudaStream_t s);

}  // namespace kda

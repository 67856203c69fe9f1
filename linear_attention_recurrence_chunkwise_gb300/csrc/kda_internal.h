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

// One unit of prefill work in task-table mode (segment-parallel forward): a
// token range of the packed tensors with its own initial and final state.
constexpr int32_t kTaskVZero = 1;       // treat v as zero over the range
constexpr int32_t kTaskS0Identity = 2;  // initial state I (d_k = d_v); S0 is ignored
constexpr int32_t kTaskNoOutput = 4;    // compute the final state only; o is not written
constexpr size_t kVZeroBytes = 64 * 128 * 2;  // one 64-token bf16 tile of a 128-wide head
struct SegTask {
    int64_t start;    // first token
    int32_t len;      // tokens
    int32_t flags;    // kTask* bits
    const float *S0;  // [H][d_v][d_k] initial state of this range, or nullptr (zeros)
    float *S_T;       // [H][d_v][d_k] final state, or nullptr (not written)
};

struct FwdParams {
    const SegTask *tasks;       // nullptr: one unit per sequence (cu_seqlens / T);
                                // else N tasks (S0 / S_T / cu_seqlens / order unused)
    const void *q, *k, *v;
    const float *log_alpha, *beta, *S0;
    const int32_t *cu_seqlens;  // nullptr: fixed length T per sequence
    void *o;
    float *S_T;
    const void *vzero;          // task mode: kVZeroBytes of zeros (the V source of
                                // kTaskVZero tasks for the tensor-core engine)
    int32_t *status;            // workspace status word
    const int32_t *order;       // workspace launch order, nullptr for fixed length
    const void *gate;           // fused output epilogue (tensor-core engine): gate
                                // logits [Ttot][H][d_v] in the io dtype, or nullptr
    const float *norm_w;        // its per-channel weight [d_v], or nullptr (ones)
    float eps;                  // its epsilon
    int blocked;                // tensor-core engine: the variant with the blocked path
                                // for chunks outside the chunk form's log-decay range
    int64_t Ttot;
    int T;                      // tokens per sequence when cu_seqlens is null
    int H, N, dk, dv;
};

// Token range of sequence (or task) n (device helper used by every prefill kernel).
__device__ __forceinline__ void seq_range(const FwdParams &p, int n, int64_t &start,
                                          int &len) {
    if (p.tasks) {
        start = p.tasks[n].start;
        len = p.tasks[n].len;
    } else if (p.cu_seqlens) {
        start = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - p.cu_seqlens[n];
    } else {
        start = (int64_t)n * p.T;
        len = p.T;
    }
}

// Where one CTA's state lives: S0 / S_T base pointers with the element offset
// of its [d_v][d_k] block and the extent the offset is checked against, plus
// the task flags (0 outside task-table mode).
struct StateRef {
    const float *S0;
    float *S_T;
    size_t off, ext;
    int32_t flags;
};

__device__ __forceinline__ StateRef state_ref(const FwdParams &p, int n, int h, int dk,
                                              int dv) {
    const size_t blk = (size_t)dk * dv;
    if (p.tasks) {
        const SegTask &t = p.tasks[n];
        return {t.S0, t.S_T, (size_t)h * blk, (size_t)p.H * blk, t.flags};
    }
    return {p.S0, p.S_T, ((size_t)n * p.H + h) * blk, (size_t)p.N * p.H * blk, 0};
}

// Initial-state element [v][c] of a CTA (identity, given or zero).
__device__ __forceinline__ float state_init(const StateRef &r, int v, int c, int dk) {
    if (r.flags & kTaskS0Identity) return v == c ? 1.f : 0.f;
    return r.S0 ? r.S0[r.off + (size_t)v * dk + c] : 0.f;
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

// Output epilogue of a KDA layer (head-wise RMSNorm times a sigmoid gate):
// y_v = sigmoid(g_v) w_v o_v / sqrt(mean_v(o_v^2) + eps) per (token, head).
// The logistic function for fp32 outputs: 1 / (1 + 2^(-x log2 e)) with the
// fast exponential and an IEEE reciprocal (relative error ~1e-7).
__device__ __forceinline__ float sigmoid_f32(float x) {
    return __frcp_rn(1.f + __expf(-x));
}
// For bf16 outputs: (1 + tanh(x / 2)) / 2 with the hardware tanh (one MUFU
// operation, absolute error about 2^-11, below the bf16 rounding of y).
__device__ __forceinline__ float sigmoid_bf16out(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
    return fmaf(0.5f, t, 0.5f);
}

// Workspace of the segment-parallel forward (byte offsets; [0, 4) is the status
// word): task tables of pass A (N (2P - 1) tasks) and pass D (N (P - 1)), the
// zero V source, and the state sets ([H][d][d] fp32 each) S_a (end of segment
// 0, per sequence), S~, M and S_in (per later segment).
struct CpLayout {
    size_t tasks_a, tasks_d, vzero, s_a, s_t, m_t, s_in, total;
};
CpLayout cp_layout(int N, int H, int d, int P);
// P >= 2 segments per sequence; base carries the validated kda_fwd arguments
// (status = the workspace).
cudaError_t launch_fwd_cp(const FwdParams &base, kda_dtype_t dt, bool use_tc, int P,
                          void *workspace, cudaStream_t s);

cudaError_t launch_schedule(const FwdParams &p, cudaStream_t s);
cudaError_t launch_prefill_simt(const FwdParams &p, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_prefill_tc(const FwdParams &p, cudaStream_t s);
bool prefill_tc_supported(kda_dtype_t dt, int dk, int dv);
// d_k = d_v = 64, fp32 or bf16 q/k/v, to fp32 accuracy (bf16 hi/lo operand pairs)
cudaError_t launch_prefill_tc64(const FwdParams &p, kda_dtype_t dt, cudaStream_t s);
// the tensor-core engine for the head size: d = 64 -> launch_prefill_tc64, else launch_prefill_tc
cudaError_t launch_prefill_tensorcore(const FwdParams &p, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_verify(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, const float *S, int N, int K, int H, int d,
                          kda_dtype_t dt, void *o, cudaStream_t s);
cudaError_t launch_commit(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, float *S, const int32_t *n_accept, int N, int K,
                          int H, int d, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *log_alpha, const float *beta, float *S, int N,
                          int H, int d, kda_dtype_t dt, void *o, cudaStream_t s,
                          const void *gate = nullptr, const float *norm_w = nullptr,
                          float eps = 0.f);
// Input prologue (ShortConv(4), Swish, L2Norm of q and k) of the three streams x[0..2]
// into y[0..2]: over whole sequences with the conv state conv0 -> conv_T (step =
// false), or one token per session with the state conv_T updated in place (step).
cudaError_t launch_short_conv(const void *const x[3], const float *const w[3], const float *conv0,
                              const int32_t *cu_seqlens, int64_t Ttot, int T, int H, int d, int N,
                              kda_dtype_t dt, float eps, void *const y[3], float *conv_T,
                              int32_t *status, bool step, cudaStream_t s);
// One token per session through the whole layer step: the input prologue from the
// projected inputs x[0..2] and the conv state (moved on in place), the decode step
// (S in place) and the output epilogue into y.
cudaError_t launch_decode_layer(const void *const x[3], const float *const w[3], float *conv,
                                float l2_eps, const float *log_alpha, const float *beta,
                                float *S, int N, int H, int d, kda_dtype_t dt, const void *gate,
                                const float *norm_w, float eps, void *y, cudaStream_t s);
// y = gated RMSNorm of o over rows of d channels (y may alias o).
cudaError_t launch_gated_rmsnorm(const void *o, const void *gate, const float *norm_w,
                                 float eps, int64_t rows, int d, kda_dtype_t dt, void *y,
                                 cudaStream_t s);

}  // namespace kda

// Fused single-token KDA decode step (CUDA cores, memory-bound).
//
// Per (session, head) the step reads the fp32 state once and writes it once:
//   Sbar[c][v] = alpha_c S[c][v]                      decay along the key axis
//   r_v        = sum_c Sbar[c][v] k_c                  old value along k
//   u_v        = beta (v_v - r_v)                      delta-rule correction
//   S'[c][v]   = Sbar[c][v] + k_c u_v                  erase + write
//   o_v        = sum_c S'[c][v] q_c = sum_c Sbar[c][v] q_c + u_v (k . q)
// which is the decode order of "Kimi Delta Attention 完全拆解" (S_decay, old_value,
// S_t, memory_output) with the read folded into the same pass over the state.
//
// Memory layout of S is [N, H, d_v, d_k]: row v holds the d_k key channels of
// value channel v contiguously.  The grid holds as many 128-thread blocks as fit
// on the GPU at once, each walking (session, head) pairs with a stride of the
// grid size (no partly filled last wave); for one pair the block
// walks rows v four at a time per warp, 8 lanes per row, every lane holding
// d/8 key channels (c = 32 i + 4 l + e), so one warp load instruction moves
// four fully used 128-byte segments.  The two k-axis reductions (r_v and the
// query read) are 3-step shuffles among the 8 lanes of a row.
//
// decode_step_gated_kernel fuses the layer's output epilogue (see there).
#include <cuda_bf16.h>

#include <atomic>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <int D, typename Tin>
__global__ void __launch_bounds__(128) decode_step_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
    const float *__restrict__ log_alpha, const float *__restrict__ beta,
    float *__restrict__ S, Tin *__restrict__ o, int NH) {
    constexpr int kLanesPerRow = 8;
    constexpr int kPerLane = D / kLanesPerRow;  // key channels per lane
    constexpr int kVec = kPerLane / 4;          // float4 per lane per row
    constexpr int kRowsPerWarp = D / 4;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane >> 3;  // row within the group of four
    const int l8 = lane & 7;

  for (int p = blockIdx.x; p < NH; p += gridDim.x) {  // (session, head) pairs
    const size_t vec = (size_t)p * D;
    float kk[kPerLane], qq[kPerLane], aa[kPerLane];
    float kq = 0.f;
#pragma unroll
    for (int i = 0; i < kVec; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 32 * i + 4 * l8 + e;
            kk[4 * i + e] = to_f(k[vec + c]);
            qq[4 * i + e] = to_f(q[vec + c]);
            aa[4 * i + e] = expf(log_alpha[vec + c]);
            kq = fmaf(kk[4 * i + e], qq[4 * i + e], kq);
        }
#pragma unroll
    for (int m = 1; m < kLanesPerRow; m <<= 1) kq += __shfl_xor_sync(0xffffffffu, kq, m);
    const float b = beta[p];
    float *Sp = S + (size_t)p * D * D;

#pragma unroll 2
    for (int r0 = warp * kRowsPerWarp; r0 < (warp + 1) * kRowsPerWarp; r0 += 4) {
        const int row = r0 + sub;
        float *Srow = Sp + (size_t)row * D + 4 * l8;
        float4 s[kVec];
#pragma unroll
        for (int i = 0; i < kVec; ++i) s[i] = *reinterpret_cast<const float4 *>(Srow + 32 * i);
        float rk = 0.f, rq = 0.f;
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
            s[i].x *= aa[4 * i + 0];
            s[i].y *= aa[4 * i + 1];
            s[i].z *= aa[4 * i + 2];
            s[i].w *= aa[4 * i + 3];
            rk = fmaf(s[i].x, kk[4 * i + 0], rk);
            rk = fmaf(s[i].y, kk[4 * i + 1], rk);
            rk = fmaf(s[i].z, kk[4 * i + 2], rk);
            rk = fmaf(s[i].w, kk[4 * i + 3], rk);
            rq = fmaf(s[i].x, qq[4 * i + 0], rq);
            rq = fmaf(s[i].y, qq[4 * i + 1], rq);
            rq = fmaf(s[i].z, qq[4 * i + 2], rq);
            rq = fmaf(s[i].w, qq[4 * i + 3], rq);
        }
#pragma unroll
        for (int m = 1; m < kLanesPerRow; m <<= 1) {
            rk += __shfl_xor_sync(0xffffffffu, rk, m);
            rq += __shfl_xor_sync(0xffffffffu, rq, m);
        }
        const float u = b * (to_f(v[vec + row]) - rk);
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
            s[i].x = fmaf(u, kk[4 * i + 0], s[i].x);
            s[i].y = fmaf(u, kk[4 * i + 1], s[i].y);
            s[i].z = fmaf(u, kk[4 * i + 2], s[i].z);
            s[i].w = fmaf(u, kk[4 * i + 3], s[i].w);
            *reinterpret_cast<float4 *>(Srow + 32 * i) = s[i];
        }
        if (l8 == 0) o[vec + row] = from_f<Tin>(fmaf(u, kq, rq));
    }
  }
}

// The same step with the layer's output epilogue fused: y_v = sigmoid(g_v)
// w_v o_v / sqrt(mean(o^2) + eps) is written instead of o (head-wise RMSNorm
// and sigmoid gate, "Kimi K3 模型结构（1）" output section).  The four warps of a
// block still split a pair's rows and never wait for one another: each posts
// its rows' outputs and the sum of their squares to a shared buffer and takes
// a ticket; the warp with the pair's last ticket writes the pair's y and
// releases the buffer.  Pairs rotate over kBufs buffers, and use u of a buffer
// (its pairs in order) owns tickets 4u .. 4u + 3.  A warp that reaches use u
// before use u - 1 of the buffer has been released -- it got kBufs pairs ahead
// of another warp -- waits for that release.  The wait always ends: the warps
// at the smallest pair index wait for a pair that every warp has passed and
// posted, whose last poster releases it without waiting (it is bounded in
// time all the same).
template <int D, typename Tin>
__global__ void __launch_bounds__(128) decode_step_gated_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
    const float *__restrict__ log_alpha, const float *__restrict__ beta,
    float *__restrict__ S, Tin *__restrict__ y, int NH, const Tin *__restrict__ gate,
    const float *__restrict__ norm_w, float eps) {
    constexpr int kLanesPerRow = 8;
    constexpr int kPerLane = D / kLanesPerRow;
    constexpr int kVec = kPerLane / 4;
    constexpr int kRowsPerWarp = D / 4;
    constexpr int kBufs = 4;
    __shared__ float o_row[kBufs][D];
    __shared__ float ss_part[kBufs][4];
    __shared__ int tickets[kBufs];   // posts to the buffer so far (4 per use)
    __shared__ int released[kBufs];  // uses of the buffer whose outputs are written

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane >> 3;
    const int l8 = lane & 7;
    if (threadIdx.x < kBufs) tickets[threadIdx.x] = released[threadIdx.x] = 0;
    __syncthreads();

  int i = 0;  // pairs this block has taken so far
  for (int p = blockIdx.x; p < NH; p += gridDim.x, ++i) {
    const int bf = i % kBufs, use = i / kBufs;
    if (lane == 0 && *reinterpret_cast<volatile int *>(&released[bf]) < use) {
        const uint64_t t0 = sm100::globaltimer_ns();
        while (*reinterpret_cast<volatile int *>(&released[bf]) < use &&
               sm100::globaltimer_ns() - t0 < sm100::kWaitLimitNs) {
        }
    }
    if (lane == 0) __threadfence_block();
    __syncwarp();
    const size_t vec = (size_t)p * D;
    float kk[kPerLane], qq[kPerLane], aa[kPerLane];
    float kq = 0.f;
#pragma unroll
    for (int i4 = 0; i4 < kVec; ++i4)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 32 * i4 + 4 * l8 + e;
            kk[4 * i4 + e] = to_f(k[vec + c]);
            qq[4 * i4 + e] = to_f(q[vec + c]);
            aa[4 * i4 + e] = expf(log_alpha[vec + c]);
            kq = fmaf(kk[4 * i4 + e], qq[4 * i4 + e], kq);
        }
#pragma unroll
    for (int m = 1; m < kLanesPerRow; m <<= 1) kq += __shfl_xor_sync(0xffffffffu, kq, m);
    const float b = beta[p];
    float *Sp = S + (size_t)p * D * D;
    float ss = 0.f;  // squares of this row group's outputs (same on its eight lanes)

#pragma unroll 2
    for (int r0 = warp * kRowsPerWarp; r0 < (warp + 1) * kRowsPerWarp; r0 += 4) {
        const int row = r0 + sub;
        float *Srow = Sp + (size_t)row * D + 4 * l8;
        float4 s[kVec];
#pragma unroll
        for (int i4 = 0; i4 < kVec; ++i4) s[i4] = *reinterpret_cast<const float4 *>(Srow + 32 * i4);
        float rk = 0.f, rq = 0.f;
#pragma unroll
        for (int i4 = 0; i4 < kVec; ++i4) {
            s[i4].x *= aa[4 * i4 + 0];
            s[i4].y *= aa[4 * i4 + 1];
            s[i4].z *= aa[4 * i4 + 2];
            s[i4].w *= aa[4 * i4 + 3];
            rk = fmaf(s[i4].x, kk[4 * i4 + 0], rk);
            rk = fmaf(s[i4].y, kk[4 * i4 + 1], rk);
            rk = fmaf(s[i4].z, kk[4 * i4 + 2], rk);
            rk = fmaf(s[i4].w, kk[4 * i4 + 3], rk);
            rq = fmaf(s[i4].x, qq[4 * i4 + 0], rq);
            rq = fmaf(s[i4].y, qq[4 * i4 + 1], rq);
            rq = fmaf(s[i4].z, qq[4 * i4 + 2], rq);
            rq = fmaf(s[i4].w, qq[4 * i4 + 3], rq);
        }
#pragma unroll
        for (int m = 1; m < kLanesPerRow; m <<= 1) {
            rk += __shfl_xor_sync(0xffffffffu, rk, m);
            rq += __shfl_xor_sync(0xffffffffu, rq, m);
        }
        const float u = b * (to_f(v[vec + row]) - rk);
#pragma unroll
        for (int i4 = 0; i4 < kVec; ++i4) {
            s[i4].x = fmaf(u, kk[4 * i4 + 0], s[i4].x);
            s[i4].y = fmaf(u, kk[4 * i4 + 1], s[i4].y);
            s[i4].z = fmaf(u, kk[4 * i4 + 2], s[i4].z);
            s[i4].w = fmaf(u, kk[4 * i4 + 3], s[i4].w);
            *reinterpret_cast<float4 *>(Srow + 32 * i4) = s[i4];
        }
        const float ov = fmaf(u, kq, rq);
        ss = fmaf(ov, ov, ss);
        if (l8 == 0) o_row[bf][row] = ov;
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 8);   // the warp's four row groups
    ss += __shfl_xor_sync(0xffffffffu, ss, 16);
    if (lane == 0) ss_part[bf][warp] = ss;
    __syncwarp();  // the warp's posts precede its count
    int last = 0;
    if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(&tickets[bf], 1) == 4 * use + 3;
        __threadfence_block();
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    __syncwarp();
    if (last) {  // every warp's posts are visible: write the pair's outputs
        const float rs = rsqrtf((ss_part[bf][0] + ss_part[bf][1] + ss_part[bf][2] +
                                 ss_part[bf][3]) * (1.f / D) + eps);
#pragma unroll
        for (int t = lane; t < D; t += 32) {
            const float gv = to_f(gate[vec + t]);
            const float sg = sizeof(Tin) == 4 ? sigmoid_f32(gv) : sigmoid_bf16out(gv);
            y[vec + t] = from_f<Tin>(o_row[bf][t] * rs * (norm_w ? norm_w[t] : 1.f) * sg);
        }
        __syncwarp();  // all lanes have read the buffer
        if (lane == 0) {
            __threadfence_block();
            atomicAdd(&released[bf], 1);
        }
    }
  }
}

template <int D, typename Tin, bool kGated>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *la,
                         const float *beta, float *S, int NH, void *o, cudaStream_t s,
                         const void *gate, const float *norm_w, float eps) {
    // resident blocks on the whole GPU, looked up once per device (threads that
    // race here all compute and store the same value)
    constexpr int kMaxDevices = 64;
    static std::atomic<int> resident[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int res = resident[dev].load(std::memory_order_relaxed);
    if (res == 0) {
        int sms = 0, per = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = kGated ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                             &per, decode_step_gated_kernel<D, Tin>, 128, 0)
                       : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                             &per, decode_step_kernel<D, Tin>, 128, 0);
        if (e != cudaSuccess) return e;
        res = sms * (per > 0 ? per : 1);
        resident[dev].store(res, std::memory_order_relaxed);
    }
    const int grid = NH < res ? NH : res;
    if constexpr (kGated)
        decode_step_gated_kernel<D, Tin><<<grid, 128, 0, s>>>(
            static_cast<const Tin *>(q), static_cast<const Tin *>(k),
                                  static_cast<const Tin *>(v), la, beta, S, static_cast<Tin *>(o),
                                  NH, static_cast<const Tin *>(gate), norm_w, eps);
    else
        decode_step_kernel<D, Tin><<<grid, 128, 0, s>>>(
            static_cast<const Tin *>(q), static_cast<const Tin *>(k),
            static_cast<const Tin *>(v), la, beta, S, static_cast<Tin *>(o), NH);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *log_alpha, const float *beta, float *S, int N,
                          int H, int d, kda_dtype_t dt, void *o, cudaStream_t s,
                          const void *gate, const float *norm_w, float eps) {
    const int NH = N * H;
    if (NH == 0) return cudaSuccess;
#define KDA_DECODE_LAUNCH(D_, T_)                                                          \
    return gate ? launch_typed<D_, T_, true>(q, k, v, log_alpha, beta, S, NH, o, s, gate,   \
                                             norm_w, eps)                                   \
                : launch_typed<D_, T_, false>(q, k, v, log_alpha, beta, S, NH, o, s, nullptr, \
                                              nullptr, 0.f)
    if (d == 128) {
        if (dt == KDA_BF16) KDA_DECODE_LAUNCH(128, __nv_bfloat16);
        KDA_DECODE_LAUNCH(128, float);
    }
    if (dt == KDA_BF16) KDA_DECODE_LAUNCH(64, __nv_bfloat16);
    KDA_DECODE_LAUNCH(64, float);
#undef KDA_DECODE_LAUNCH
}

}  // namespace kda

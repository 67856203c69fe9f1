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
#include <cuda_bf16.h>

#include <atomic>

#include "kda_internal.h"

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

template <int D, typename Tin>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *la,
                         const float *beta, float *S, int NH, void *o, cudaStream_t s) {
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
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, decode_step_kernel<D, Tin>,
                                                              128, 0);
        if (e != cudaSuccess) return e;
        res = sms * (per > 0 ? per : 1);
        resident[dev].store(res, std::memory_order_relaxed);
    }
    const int grid = NH < res ? NH : res;
    decode_step_kernel<D, Tin><<<grid, 128, 0, s>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k),
        static_cast<const Tin *>(v), la, beta, S, static_cast<Tin *>(o), NH);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const float *log_alpha, const float *beta, float *S, int N,
                          int H, int d, kda_dtype_t dt, void *o, cudaStream_t s) {
    const int NH = N * H;
    if (NH == 0) return cudaSuccess;
    if (d == 128)
        return dt == KDA_BF16
                   ? launch_typed<128, __nv_bfloat16>(q, k, v, log_alpha, beta, S, NH, o, s)
                   : launch_typed<128, float>(q, k, v, log_alpha, beta, S, NH, o, s);
    return dt == KDA_BF16
               ? launch_typed<64, __nv_bfloat16>(q, k, v, log_alpha, beta, S, NH, o, s)
               : launch_typed<64, float>(q, k, v, log_alpha, beta, S, NH, o, s);
}

}  // namespace kda

// Output epilogue of a KDA layer as a pass of its own: per (token, head) row of
// d value channels, y = sigmoid(g) w o / sqrt(mean(o^2) + eps) -- the head-wise
// RMSNorm over the value channels and the sigmoid output gate of "Kimi K3 模型
// 结构（1）" (output section) and "Kimi K3模型架构详解" section 3.2.  The
// tensor-core prefill and the decode step fuse the same arithmetic into their
// output stores; this kernel serves the CUDA-core prefill engine and callers
// that hold o already.  Memory-bound: one warp per row, o and g read once, y
// written once (y may alias o: each warp reads its whole row before writing).
#include <cuda_bf16.h>

#include <atomic>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

template <int D>
__device__ __forceinline__ void load_row(const float *p, float (&x)[D / 32]) {
    if constexpr (D == 128) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w;
    } else {
        const float2 a = *reinterpret_cast<const float2 *>(p);
        x[0] = a.x, x[1] = a.y;
    }
}
template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *p, float (&x)[D / 32]) {
    if constexpr (D == 128) {
        const uint2 a = *reinterpret_cast<const uint2 *>(p);
        x[0] = __uint_as_float(a.x << 16), x[1] = __uint_as_float(a.x & 0xFFFF0000u);
        x[2] = __uint_as_float(a.y << 16), x[3] = __uint_as_float(a.y & 0xFFFF0000u);
    } else {
        const uint32_t a = *reinterpret_cast<const uint32_t *>(p);
        x[0] = __uint_as_float(a << 16), x[1] = __uint_as_float(a & 0xFFFF0000u);
    }
}
template <int D>
__device__ __forceinline__ void store_row(float *p, const float (&y)[D / 32]) {
    if constexpr (D == 128)
        *reinterpret_cast<float4 *>(p) = make_float4(y[0], y[1], y[2], y[3]);
    else
        *reinterpret_cast<float2 *>(p) = make_float2(y[0], y[1]);
}
template <int D>
__device__ __forceinline__ void store_row(__nv_bfloat16 *p, const float (&y)[D / 32]) {
    const uint32_t lo = sm100::pack_bf16(y[0], y[1]);
    if constexpr (D == 128)
        *reinterpret_cast<uint2 *>(p) = make_uint2(lo, sm100::pack_bf16(y[2], y[3]));
    else
        *reinterpret_cast<uint32_t *>(p) = lo;
}

template <int D, typename T>
__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(const T *o, const T *__restrict__ g,
                                                            const float *__restrict__ w,
                                                            float eps, int64_t rows, T *y) {
    constexpr int E = D / 32;  // channels per lane, contiguous
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    float wl[E];
#pragma unroll
    for (int e = 0; e < E; ++e) wl[e] = w ? w[E * lane + e] : 1.f;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
         r += nwarps) {
        const size_t off = (size_t)r * D + E * lane;
        float x[E], gg[E];
        load_row<D>(o + off, x);
        load_row<D>(g + off, gg);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float rs = rsqrtf(ss * (1.f / D) + eps);
        float yy[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float sg = sizeof(T) == 4 ? sigmoid_f32(gg[e]) : sigmoid_bf16out(gg[e]);
            yy[e] = x[e] * rs * wl[e] * sg;
        }
        store_row<D>(y + off, yy);
    }
}

template <int D, typename T>
cudaError_t launch_typed(const void *o, const void *g, const float *w, float eps, int64_t rows,
                         void *y, cudaStream_t s) {
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
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, gated_rmsnorm_kernel<D, T>,
                                                              256, 0);
        if (e != cudaSuccess) return e;
        res = sms * (per > 0 ? per : 1);
        resident[dev].store(res, std::memory_order_relaxed);
    }
    const int64_t need = (rows + 7) / 8;  // 8 rows (warps) per block
    const int grid = (int)(need < res ? need : res);
    gated_rmsnorm_kernel<D, T><<<grid, 256, 0, s>>>(static_cast<const T *>(o),
                                                    static_cast<const T *>(g), w, eps, rows,
                                                    static_cast<T *>(y));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const void *o, const void *gate, const float *norm_w,
                                 float eps, int64_t rows, int d, kda_dtype_t dt, void *y,
                                 cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    if (d == 128)
        return dt == KDA_BF16 ? launch_typed<128, __nv_bfloat16>(o, gate, norm_w, eps, rows, y, s)
                              : launch_typed<128, float>(o, gate, norm_w, eps, rows, y, s);
    return dt == KDA_BF16 ? launch_typed<64, __nv_bfloat16>(o, gate, norm_w, eps, rows, y, s)
                          : launch_typed<64, float>(o, gate, norm_w, eps, rows, y, s);
}

}  // namespace kda

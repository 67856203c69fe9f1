// Speculative-decode verification and commit over K cached draft tokens
// ("Kimi K3 深度拆解" section 9.2: the inference kernel keeps the draft
// tokens' projected inputs instead of a copy of the state per draft position,
// and after verification replays the accepted tokens on chip to rebuild the
// state it writes back).
//
//   verify: from the committed state S, the outputs of K consecutive draft
//           tokens per session; S is read once and left as it is.
//   commit: the first n_accept[n] of the same cached tokens applied to S in
//           place; S is read and written once.
//
// Every value channel v evolves on its own through the decode recurrence
// (decay along c, old_v = sum_c Sbar[c][v] k_c, u_v = beta (v_v - old_v),
// S'[c][v] = Sbar[c][v] + k_c u_v, o_v = sum_c S'[c][v] q_c), so a row v of
// the [d_v][d_k] state stays in registers while it runs through all the
// tokens.  The lane layout, the per-token arithmetic and its summation order
// are those of the single-token decode kernel, so K calls of kda_decode_step
// and one verify / commit give the same numbers.
//
// One 128-thread block per (session, head) at a time (a grid of the resident
// blocks walks the pairs).  The K tokens' k, q, alpha = exp(log_alpha) and v
// are staged in shared memory first, with k . q per token computed once.
#include <cuda_bf16.h>

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

template <int D>
struct MtSmem {
    float k[KDA_MAX_DRAFT_TOKENS][D], q[KDA_MAX_DRAFT_TOKENS][D];
    float a[KDA_MAX_DRAFT_TOKENS][D], v[KDA_MAX_DRAFT_TOKENS][D];
    float beta[KDA_MAX_DRAFT_TOKENS], kq[KDA_MAX_DRAFT_TOKENS];
};

template <int D, typename Tin, bool kCommit>
__global__ void __launch_bounds__(128) multi_token_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
    const float *__restrict__ log_alpha, const float *__restrict__ beta, float *__restrict__ S,
    const int32_t *__restrict__ n_accept, Tin *__restrict__ o, int N, int K, int H) {
    constexpr int kLanesPerRow = 8;
    constexpr int kPerLane = D / kLanesPerRow;  // key channels per lane
    constexpr int kVec = kPerLane / 4;          // float4 per lane per row
    constexpr int kRowsPerWarp = D / 4;
    __shared__ MtSmem<D> sm;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane >> 3;  // row within the group of four
    const int l8 = lane & 7;

    for (int p = blockIdx.x; p < N * H; p += gridDim.x) {  // (session, head) pairs
        const int n = p / H, h = p % H;
        int steps = K;
        if (kCommit && n_accept) steps = min(max(n_accept[n], 0), K);
        __syncthreads();  // the previous pair is done with the staged tokens
        for (int i = threadIdx.x; i < K * D; i += blockDim.x) {
            const int t = i / D, c = i % D;
            const size_t g = ((size_t)(n * K + t) * H + h) * D + c;
            sm.k[t][c] = to_f(k[g]);
            sm.a[t][c] = expf(log_alpha[g]);
            sm.v[t][c] = to_f(v[g]);
            if (!kCommit) sm.q[t][c] = to_f(q[g]);
        }
        if (threadIdx.x < K) sm.beta[threadIdx.x] = beta[(size_t)(n * K + threadIdx.x) * H + h];
        __syncthreads();
        if (!kCommit && warp == 0) {  // k . q per token, in the decode kernel's order
            for (int t = 0; t < K; ++t) {
                float kq = 0.f;
#pragma unroll
                for (int i = 0; i < kVec; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 32 * i + 4 * l8 + e;
                        kq = fmaf(sm.k[t][c], sm.q[t][c], kq);
                    }
#pragma unroll
                for (int m = 1; m < kLanesPerRow; m <<= 1) kq += __shfl_xor_sync(0xffffffffu, kq, m);
                if (lane == 0) sm.kq[t] = kq;
            }
        }
        __syncthreads();
        if (kCommit && steps == 0) continue;  // nothing accepted: S stays as it is

        float *Sp = S + (size_t)p * D * D;
        for (int r0 = warp * kRowsPerWarp; r0 < (warp + 1) * kRowsPerWarp; r0 += 4) {
            const int row = r0 + sub;
            float *Srow = Sp + (size_t)row * D + 4 * l8;
            float4 s[kVec];
#pragma unroll
            for (int i = 0; i < kVec; ++i) s[i] = *reinterpret_cast<const float4 *>(Srow + 32 * i);
            for (int t = 0; t < steps; ++t) {
                const float *kt = sm.k[t] + 4 * l8, *at = sm.a[t] + 4 * l8, *qt = sm.q[t] + 4 * l8;
                float kk[kPerLane];
                float rk = 0.f, rq = 0.f;
#pragma unroll
                for (int i = 0; i < kVec; ++i) {
                    const float4 ka = *reinterpret_cast<const float4 *>(kt + 32 * i);
                    const float4 aa = *reinterpret_cast<const float4 *>(at + 32 * i);
                    kk[4 * i] = ka.x, kk[4 * i + 1] = ka.y, kk[4 * i + 2] = ka.z, kk[4 * i + 3] = ka.w;
                    s[i].x *= aa.x;
                    s[i].y *= aa.y;
                    s[i].z *= aa.z;
                    s[i].w *= aa.w;
                    rk = fmaf(s[i].x, ka.x, rk);
                    rk = fmaf(s[i].y, ka.y, rk);
                    rk = fmaf(s[i].z, ka.z, rk);
                    rk = fmaf(s[i].w, ka.w, rk);
                    if (!kCommit) {
                        const float4 qa = *reinterpret_cast<const float4 *>(qt + 32 * i);
                        rq = fmaf(s[i].x, qa.x, rq);
                        rq = fmaf(s[i].y, qa.y, rq);
                        rq = fmaf(s[i].z, qa.z, rq);
                        rq = fmaf(s[i].w, qa.w, rq);
                    }
                }
#pragma unroll
                for (int m = 1; m < kLanesPerRow; m <<= 1) {
                    rk += __shfl_xor_sync(0xffffffffu, rk, m);
                    if (!kCommit) rq += __shfl_xor_sync(0xffffffffu, rq, m);
                }
                const float u = sm.beta[t] * (sm.v[t][row] - rk);
#pragma unroll
                for (int i = 0; i < kVec; ++i) {
                    s[i].x = fmaf(u, kk[4 * i + 0], s[i].x);
                    s[i].y = fmaf(u, kk[4 * i + 1], s[i].y);
                    s[i].z = fmaf(u, kk[4 * i + 2], s[i].z);
                    s[i].w = fmaf(u, kk[4 * i + 3], s[i].w);
                }
                if (!kCommit && l8 == 0)
                    o[((size_t)(n * K + t) * H + h) * D + row] = from_f<Tin>(fmaf(u, sm.kq[t], rq));
            }
            if (kCommit) {
#pragma unroll
                for (int i = 0; i < kVec; ++i) *reinterpret_cast<float4 *>(Srow + 32 * i) = s[i];
            }
        }
    }
}

template <int D, typename Tin, bool kCommit>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *la,
                         const float *beta, float *S, const int32_t *n_accept, void *o, int N,
                         int K, int H, cudaStream_t s) {
    constexpr int kMaxDevices = 64;
    static int resident[kMaxDevices];  // every thread that races here computes the same value
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (resident[dev] == 0) {
        int sms = 0, per = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per, multi_token_kernel<D, Tin, kCommit>, 128, 0);
        if (e != cudaSuccess) return e;
        resident[dev] = sms * (per > 0 ? per : 1);
    }
    const int pairs = N * H;
    const int grid = pairs < resident[dev] ? pairs : resident[dev];
    multi_token_kernel<D, Tin, kCommit><<<grid, 128, 0, s>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        la, beta, S, n_accept, static_cast<Tin *>(o), N, K, H);
    return cudaGetLastError();
}

template <bool kCommit>
cudaError_t launch_dispatch(const void *q, const void *k, const void *v, const float *la,
                            const float *beta, float *S, const int32_t *n_accept, void *o,
                            int N, int K, int H, int d, kda_dtype_t dt, cudaStream_t s) {
    if (d == 128)
        return dt == KDA_BF16
                   ? launch_typed<128, __nv_bfloat16, kCommit>(q, k, v, la, beta, S, n_accept,
                                                               o, N, K, H, s)
                   : launch_typed<128, float, kCommit>(q, k, v, la, beta, S, n_accept, o, N,
                                                       K, H, s);
    return dt == KDA_BF16
               ? launch_typed<64, __nv_bfloat16, kCommit>(q, k, v, la, beta, S, n_accept, o,
                                                          N, K, H, s)
               : launch_typed<64, float, kCommit>(q, k, v, la, beta, S, n_accept, o, N, K, H,
                                                  s);
}

}  // namespace

cudaError_t launch_verify(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, const float *S, int N, int K, int H, int d,
                          kda_dtype_t dt, void *o, cudaStream_t s) {
    if ((size_t)N * H == 0) return cudaSuccess;
    return launch_dispatch<false>(q, k, v, log_alpha, beta, const_cast<float *>(S), nullptr,
                                  o, N, K, H, d, dt, s);
}

cudaError_t launch_commit(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, float *S, const int32_t *n_accept, int N, int K,
                          int H, int d, kda_dtype_t dt, cudaStream_t s) {
    if ((size_t)N * H == 0) return cudaSuccess;
    return launch_dispatch<true>(q, k, v, log_alpha, beta, S, n_accept, nullptr, N, K, H, d,
                                 dt, s);
}

}  // namespace kda

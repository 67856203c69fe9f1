// Input prologue of a KDA layer: q, k = L2Norm(Swish(ShortConv(W x))), v =
// Swish(ShortConv(W_v x)) ("Kimi Delta Attention 完全拆解", the KDA layer's
// forward; "Kimi K3 模型结构（1）", parameterisation section: a depthwise causal
// convolution of kernel 4 along the sequence that mixes each token with the
// three before it, and the last three projected inputs of q, k, v kept for
// decode as the layer's only state besides S).  Per channel, with taps w[0..3]
// (w[3] on the current token) and x_{-3..-1} taken from the conv state:
//   c_t = w[0] x_{t-3} + w[1] x_{t-2} + w[2] x_{t-1} + w[3] x_t,
//   y_t = c_t sigmoid(c_t),   q, k: y_t / sqrt(sum_d y_t^2 + eps) per (token, head).
//
// A memory-bound pass: one warp per (stream, head, run of 64 packed tokens),
// lane l holding channels d/32 l .. d/32 (l + 1) - 1 of each row, the three
// previous inputs in registers as the window slides,
// the L2 norm's sum by a warp butterfly.  Consecutive warps take consecutive
// heads of the same tokens, so the rows they read are neighbours in memory.
// A run that crosses into another sequence reloads its window there; windows
// before a sequence's first token come from the caller's conv state (zeros
// without one).  A second small pass writes the final conv state, so that it
// may overwrite the initial one in place.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kRun = 64;    // tokens per warp
constexpr int kWarps = 8;   // warps per block

struct ConvParams {
    const void *x[3];        // xq, xk, xv  [Ttot][H][D]
    const float *w[3];       // taps        [H][D][4]
    const float *conv0;      // [N][3][3][H][D] or nullptr
    const int32_t *cu;       // [N + 1] or nullptr (fixed length T)
    void *y[3];              // q, k, v     [Ttot][H][D]
    float *conv_T;           // [N][3][3][H][D] or nullptr
    int32_t *status;
    int64_t Ttot;
    int T, H, N;
    float eps;
};

__device__ __forceinline__ float ld1(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld1(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}

// kC consecutive elements from element index i (this lane's channels of one
// row), as one vector load
template <int kC, typename T>
__device__ __forceinline__ void load_lane(const T *p, size_t i, float (&f)[kC]) {
    if constexpr (sizeof(T) == 4 && kC == 4) {
        const float4 a = *reinterpret_cast<const float4 *>(p + i);
        f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w;
    } else if constexpr (sizeof(T) == 4 && kC == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(p + i);
        f[0] = a.x, f[1] = a.y;
    } else if constexpr (kC == 4) {  // bf16
        const uint2 a = *reinterpret_cast<const uint2 *>(p + i);
        f[0] = __uint_as_float(a.x << 16), f[1] = __uint_as_float(a.x & 0xFFFF0000u);
        f[2] = __uint_as_float(a.y << 16), f[3] = __uint_as_float(a.y & 0xFFFF0000u);
    } else {
        const uint32_t a = *reinterpret_cast<const uint32_t *>(p + i);
        f[0] = __uint_as_float(a << 16), f[1] = __uint_as_float(a & 0xFFFF0000u);
    }
}

template <int kC, typename T>
__device__ __forceinline__ void store_lane(T *p, size_t i, const float (&f)[kC]) {
    if constexpr (sizeof(T) == 4 && kC == 4) {
        *reinterpret_cast<float4 *>(p + i) = make_float4(f[0], f[1], f[2], f[3]);
    } else if constexpr (sizeof(T) == 4 && kC == 2) {
        *reinterpret_cast<float2 *>(p + i) = make_float2(f[0], f[1]);
    } else {
        __nv_bfloat16 b[kC];
#pragma unroll
        for (int e = 0; e < kC; ++e) b[e] = __float2bfloat16_rn(f[e]);
        if constexpr (kC == 4) {
            uint2 u;
            u.x = (uint32_t)__bfloat16_as_ushort(b[0]) | ((uint32_t)__bfloat16_as_ushort(b[1]) << 16);
            u.y = (uint32_t)__bfloat16_as_ushort(b[2]) | ((uint32_t)__bfloat16_as_ushort(b[3]) << 16);
            *reinterpret_cast<uint2 *>(p + i) = u;
        } else {
            *reinterpret_cast<uint32_t *>(p + i) =
                (uint32_t)__bfloat16_as_ushort(b[0]) | ((uint32_t)__bfloat16_as_ushort(b[1]) << 16);
        }
    }
}

// ShortConv + Swish (+ L2Norm) of one row from the window and the current input.
// The pass is bound by its instruction count, so the sigmoid is taken as
// 1 / (1 + 2^(-c log2 e)) with the fast exponential and division (a few ulp)
// for fp32 outputs, and as (1 + tanh(c / 2)) / 2 with the hardware tanh (about
// 2^-11, below the output's own rounding) for bf16 outputs.
template <int kC, bool kBf16Out>
__device__ __forceinline__ void conv_row(const float (&w)[kC][4], const float (&win)[3][kC],
                                         const float (&xt)[kC], bool norm, float eps,
                                         float (&y)[kC]) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < kC; ++e) {
        float c = w[e][3] * xt[e];
        c = fmaf(w[e][2], win[2][e], c);
        c = fmaf(w[e][1], win[1][e], c);
        c = fmaf(w[e][0], win[0][e], c);
        y[e] = kBf16Out ? c * sigmoid_bf16out(c) : __fdividef(c, 1.f + __expf(-c));
        ss = fmaf(y[e], y[e], ss);
    }
    if (norm) {
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float t = ss + eps;
        const float r = t > 0.f ? rsqrtf(t) : 0.f;
#pragma unroll
        for (int e = 0; e < kC; ++e) y[e] *= r;
    }
}

// the sequence holding packed token t: cu[n] <= t < cu[n + 1] (empty sequences
// skipped: the last n with cu[n] <= t)
__device__ __forceinline__ int seq_of(const ConvParams &p, int64_t t) {
    if (!p.cu) return (int)(t / p.T);
    int lo = 0, hi = p.N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int64_t seq_start(const ConvParams &p, int n) {
    return p.cu ? (int64_t)p.cu[n] : (int64_t)n * p.T;
}

template <int kBytes>
__device__ __forceinline__ void cp_async(void *dst, const void *src) {
    if constexpr (kBytes == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src), "n"(kBytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int n>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory"); }

// Rows are staged in shared memory by cp.async, eight at a time and double
// buffered: the next eight rows are in flight while the current ones are
// computed, without holding registers (rows loaded into registers, two or four
// at a time, kept the pass at 0.5 of the copy bandwidth: too few bytes in
// flight per SM).  Each lane copies, and reads back, only its own piece of a
// row, so no barrier is needed.
constexpr int kAsyncGroup = 8;

template <int D, typename T>
__global__ void __launch_bounds__(32 * kWarps) short_conv_kernel(const __grid_constant__ ConvParams p) {
    constexpr int kC = D / 32;
    constexpr int kLane = kC * (int)sizeof(T);      // bytes of one row held by a lane
    constexpr int kBuf = kAsyncGroup * 32 * kLane;  // one group of rows of one warp
    extern __shared__ __align__(16) uint8_t stage_raw[];
    if (*p.status == KDA_ERR_INVALID_ARGUMENT) return;  // set by the schedule kernel
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint8_t *stage = stage_raw + wid * 2 * kBuf + lane * kLane;  // this lane's pieces
    const int64_t gw = (int64_t)blockIdx.x * kWarps + wid;
    const int64_t nruns = (p.Ttot + kRun - 1) / kRun;
    const int64_t per_stream = nruns * p.H;
    if (gw >= 3 * per_stream) return;
    const int s = (int)(gw / per_stream);
    const int64_t rem = gw % per_stream;
    const int h = (int)(rem % p.H);
    const int64_t t_begin = (rem / p.H) * kRun, t_end = min(p.Ttot, t_begin + kRun);
    const T *x = static_cast<const T *>(p.x[s]);
    T *y = static_cast<T *>(p.y[s]);
    const bool norm = s < 2;
    const size_t n_tok = (size_t)p.Ttot * p.H * D, n_state = (size_t)p.N * 9 * p.H * D;
    const int c0 = kC * lane;
    float w[kC][4];
#pragma unroll
    for (int e = 0; e < kC; ++e) {
        const float4 t4 = *reinterpret_cast<const float4 *>(p.w[s] + ((size_t)h * D + c0 + e) * 4);
        w[e][0] = t4.x, w[e][1] = t4.y, w[e][2] = t4.z, w[e][3] = t4.w;
    }
    int n = seq_of(p, t_begin);
    int64_t start = seq_start(p, n), end = seq_start(p, n + 1);
    float win[3][kC] = {};
    auto load_window = [&](int64_t t) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int64_t q = t - 3 + j;
            if (q >= start) {
                const size_t i = ((size_t)q * p.H + h) * D + c0;
                if (in_bounds(p.status, i + kC - 1, n_tok)) load_lane<kC>(x, i, win[j]);
            } else if (p.conv0) {
                const size_t i = ((((size_t)n * 3 + s) * 3 + (size_t)(q - start + 3)) * p.H + h) * D + c0;
                if (in_bounds(p.status, i + kC - 1, n_state)) load_lane<kC>(p.conv0, i, win[j]);
            } else {
#pragma unroll
                for (int e = 0; e < kC; ++e) win[j][e] = 0.f;
            }
        }
    };
    // rows of group g -> buffer g % 2 (each lane copies, and later reads back,
    // only its own piece of each row)
    auto prefetch = [&](int64_t tg, int buf) {
#pragma unroll
        for (int g = 0; g < kAsyncGroup; ++g) {
            const size_t i = ((size_t)(tg + g) * p.H + h) * D + c0;
            if (tg + g < t_end && in_bounds(p.status, i + kC - 1, n_tok))
                cp_async<kLane>(stage + buf * kBuf + g * 32 * kLane, x + i);
        }
        cp_commit();
    };
    load_window(t_begin);
    prefetch(t_begin, 0);
    int buf = 0;
    for (int64_t tg = t_begin; tg < t_end; tg += kAsyncGroup, buf ^= 1) {
        if (tg + kAsyncGroup < t_end) {
            prefetch(tg + kAsyncGroup, buf ^ 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        const uint8_t *rows = stage + buf * kBuf;
        if (tg + kAsyncGroup <= t_end && tg + kAsyncGroup <= end) {
            // the whole group inside the current sequence: no branches; the
            // L2 norms of its eight tokens from one reduce-scatter of their
            // partial sums (lane l ends with token (l >> 2) & 7's total) and
            // eight shuffles back, in place of a butterfly per token
            T *yp = y + ((size_t)tg * p.H + h) * D + c0;
            const size_t step = (size_t)p.H * D;
            float yg[kAsyncGroup][kC], ss[kAsyncGroup];
#pragma unroll
            for (int g = 0; g < kAsyncGroup; ++g) {
                float xt[kC];
                load_lane<kC>(reinterpret_cast<const T *>(rows + g * 32 * kLane), 0, xt);
                conv_row<kC, sizeof(T) == 2>(w, win, xt, false, 0.f, yg[g]);
                ss[g] = 0.f;
#pragma unroll
                for (int e = 0; e < kC; ++e) {
                    ss[g] = fmaf(yg[g][e], yg[g][e], ss[g]);
                    win[0][e] = win[1][e];
                    win[1][e] = win[2][e];
                    win[2][e] = xt[e];
                }
            }
            if (norm) {
#pragma unroll
                for (int len = 4; len >= 1; len >>= 1) {  // lane bits 4, 3, 2 halve the set
                    const bool up = lane & (4 * len);
#pragma unroll
                    for (int i = 0; i < len; ++i) {
                        const float keep = up ? ss[i + len] : ss[i];
                        const float send = up ? ss[i] : ss[i + len];
                        ss[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4 * len);
                    }
                }
                ss[0] += __shfl_xor_sync(0xffffffffu, ss[0], 2);
                ss[0] += __shfl_xor_sync(0xffffffffu, ss[0], 1);
                const float t = ss[0] + p.eps;
                const float r = t > 0.f ? rsqrtf(t) : 0.f;
#pragma unroll
                for (int g = 0; g < kAsyncGroup; ++g) {
                    const float rg = __shfl_sync(0xffffffffu, r, 4 * g);
#pragma unroll
                    for (int e = 0; e < kC; ++e) yg[g][e] *= rg;
                }
            }
#pragma unroll
            for (int g = 0; g < kAsyncGroup; ++g)
                if (in_bounds(p.status, ((size_t)(tg + g) * p.H + h) * D + c0 + kC - 1, n_tok))
                    store_lane<kC>(yp + g * step, 0, yg[g]);
            continue;
        }
#pragma unroll
        for (int g = 0; g < kAsyncGroup; ++g) {
            const int64_t t = tg + g;
            if (t >= t_end) break;
            if (t == end) {  // the run enters the next non-empty sequence
                while (seq_start(p, n + 1) <= t) ++n;
                start = seq_start(p, n);
                end = seq_start(p, n + 1);
                load_window(t);
            }
            float xt[kC], yv[kC];
            load_lane<kC>(reinterpret_cast<const T *>(stage + buf * kBuf + g * 32 * kLane), 0, xt);
            conv_row<kC, sizeof(T) == 2>(w, win, xt, norm, p.eps, yv);
            const size_t i = ((size_t)t * p.H + h) * D + c0;
            if (in_bounds(p.status, i + kC - 1, n_tok)) store_lane<kC>(y, i, yv);
#pragma unroll
            for (int e = 0; e < kC; ++e) {
                win[0][e] = win[1][e];
                win[1][e] = win[2][e];
                win[2][e] = xt[e];
            }
        }
    }
}

// final conv state: per (sequence, stream, head, channel) the last three inputs
// (with the initial state's tail for a sequence shorter than three), all read
// before any is written, so conv_T may be conv0
template <int D, typename T>
__global__ void conv_state_kernel(const __grid_constant__ ConvParams p) {
    if (*p.status == KDA_ERR_INVALID_ARGUMENT) return;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)p.N * 3 * p.H * D;
    if (idx >= total) return;
    const int c = (int)(idx % D);
    const int h = (int)((idx / D) % p.H);
    const int s = (int)((idx / ((size_t)D * p.H)) % 3);
    const int n = (int)(idx / ((size_t)3 * p.H * D));
    const int64_t start = seq_start(p, n), len = seq_start(p, n + 1) - start;
    const T *x = static_cast<const T *>(p.x[s]);
    const size_t n_tok = (size_t)p.Ttot * p.H * D, n_state = (size_t)p.N * 9 * p.H * D;
    float v[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int64_t q = len - 3 + j;
        v[j] = 0.f;
        if (q >= 0) {
            const size_t i = ((size_t)(start + q) * p.H + h) * D + c;
            if (in_bounds(p.status, i, n_tok)) v[j] = ld1(x, i);
        } else if (p.conv0) {
            const size_t i = ((((size_t)n * 3 + s) * 3 + (size_t)(q + 3)) * p.H + h) * D + c;
            if (in_bounds(p.status, i, n_state)) v[j] = p.conv0[i];
        }
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const size_t i = ((((size_t)n * 3 + s) * 3 + j) * p.H + h) * D + c;
        if (in_bounds(p.status, i, n_state)) p.conv_T[i] = v[j];
    }
}

// one token per session: warp per (session, stream, head); the conv state
// [N][3][3][H][D] is read, then shifted by one token in place
template <int D, typename T>
__global__ void __launch_bounds__(32 * kWarps) short_conv_step_kernel(const __grid_constant__ ConvParams p) {
    constexpr int kC = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (gw >= (int64_t)p.N * 3 * p.H) return;
    const int h = (int)(gw % p.H);
    const int s = (int)((gw / p.H) % 3);
    const int n = (int)(gw / ((int64_t)3 * p.H));
    const int c0 = kC * lane;
    const size_t n_tok = (size_t)p.N * p.H * D, n_state = (size_t)p.N * 9 * p.H * D;
    float w[kC][4];
#pragma unroll
    for (int e = 0; e < kC; ++e) {
        const float4 t4 = *reinterpret_cast<const float4 *>(p.w[s] + ((size_t)h * D + c0 + e) * 4);
        w[e][0] = t4.x, w[e][1] = t4.y, w[e][2] = t4.z, w[e][3] = t4.w;
    }
    float win[3][kC] = {}, xt[kC] = {}, yv[kC];
    size_t si[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        si[j] = ((((size_t)n * 3 + s) * 3 + j) * p.H + h) * D + c0;
        if (in_bounds(p.status, si[j] + kC - 1, n_state)) load_lane<kC>(p.conv_T, si[j], win[j]);
    }
    const size_t i = ((size_t)n * p.H + h) * D + c0;
    if (in_bounds(p.status, i + kC - 1, n_tok)) load_lane<kC>(static_cast<const T *>(p.x[s]), i, xt);
    conv_row<kC, sizeof(T) == 2>(w, win, xt, s < 2, p.eps, yv);
    if (in_bounds(p.status, i + kC - 1, n_tok)) store_lane<kC>(static_cast<T *>(p.y[s]), i, yv);
    // the window moves on by one token: (x_{t-2}, x_{t-1}, x_t)
    if (in_bounds(p.status, si[0] + kC - 1, n_state)) store_lane<kC>(p.conv_T, si[0], win[1]);
    if (in_bounds(p.status, si[1] + kC - 1, n_state)) store_lane<kC>(p.conv_T, si[1], win[2]);
    if (in_bounds(p.status, si[2] + kC - 1, n_state)) store_lane<kC>(p.conv_T, si[2], xt);
}

template <int D, typename T>
cudaError_t launch_typed(const ConvParams &p, bool step, cudaStream_t s) {
    if (step) {
        const int64_t warps = (int64_t)p.N * 3 * p.H;
        if (warps == 0) return cudaSuccess;
        short_conv_step_kernel<D, T><<<(unsigned)((warps + kWarps - 1) / kWarps), 32 * kWarps, 0, s>>>(p);
        return cudaGetLastError();
    }
    const int64_t warps = 3 * ((p.Ttot + kRun - 1) / kRun) * p.H;
    const int smem = kWarps * 2 * kAsyncGroup * D * (int)sizeof(T);
    if (warps > 0) {
        cudaError_t e0 = cudaFuncSetAttribute(short_conv_kernel<D, T>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e0 != cudaSuccess) return e0;
        short_conv_kernel<D, T><<<(unsigned)((warps + kWarps - 1) / kWarps), 32 * kWarps, smem, s>>>(p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !p.conv_T) return e;
    const size_t total = (size_t)p.N * 3 * p.H * D;
    if (total == 0) return cudaSuccess;
    conv_state_kernel<D, T><<<(unsigned)((total + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_short_conv(const void *const x[3], const float *const w[3], const float *conv0,
                              const int32_t *cu_seqlens, int64_t Ttot, int T, int H, int d, int N,
                              kda_dtype_t dt, float eps, void *const y[3], float *conv_T,
                              int32_t *status, bool step, cudaStream_t s) {
    ConvParams p{};
    for (int i = 0; i < 3; ++i) {
        p.x[i] = x[i];
        p.w[i] = w[i];
        p.y[i] = y[i];
    }
    p.conv0 = conv0;
    p.cu = cu_seqlens;
    p.conv_T = conv_T;
    p.status = status;
    p.Ttot = Ttot;
    p.T = T;
    p.H = H;
    p.N = N;
    p.eps = eps;
    if (d == 128)
        return dt == KDA_F32 ? launch_typed<128, float>(p, step, s)
                             : launch_typed<128, __nv_bfloat16>(p, step, s);
    return dt == KDA_F32 ? launch_typed<64, float>(p, step, s)
                         : launch_typed<64, __nv_bfloat16>(p, step, s);
}

}  // namespace kda

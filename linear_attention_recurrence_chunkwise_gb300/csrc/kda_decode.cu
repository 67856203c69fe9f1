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

// The layer's input prologue computed in the step (kPro): q, k = L2Norm(Swish(
// ShortConv(x))), v = Swish(ShortConv(x_v)) from the projected inputs x of the
// session's token and the conv state (the three previous inputs per stream),
// which the step then moves on by one token ("Kimi K3" (gentlecold) section 9.2:
// the inference kernel fuses the short convolution, the input normalisation,
// the recurrence and the output normalisation; the prologue's arithmetic is
// the one kda_short_conv_step runs).
struct PrologueArgs {
    const void *x[3];  // xq, xk, xv [N][H][D]
    const float *w[3];  // taps [H][D][4], w[3] on the current token
    float *conv;        // [N][3][3][H][D], updated in place
    int H;
    float l2_eps;
};

__device__ __forceinline__ float swish(float c, bool bf16_out) {
    return bf16_out ? c * sigmoid_bf16out(c) : __fdividef(c, 1.f + __expf(-c));
}

// four consecutive elements of an input row as floats
__device__ __forceinline__ void load4(const float *p, size_t i, float (&f)[4]) {
    const float4 a = *reinterpret_cast<const float4 *>(p + i);
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, size_t i, float (&f)[4]) {
    const uint2 a = *reinterpret_cast<const uint2 *>(p + i);
    f[0] = __uint_as_float(a.x << 16), f[1] = __uint_as_float(a.x & 0xFFFF0000u);
    f[2] = __uint_as_float(a.y << 16), f[3] = __uint_as_float(a.y & 0xFFFF0000u);
}

// q or k (stream s) of pair (n, h) on this lane's channels c = 32 i + 4 l8 + e.
// The four row groups of the warp hold the same channels, so row group `sub`
// computes slice i = sub (four channels per lane) and the lanes gather the
// other slices by shuffles; the L2 norm's sum runs over the whole warp.
template <int D, typename Tin>
__device__ __forceinline__ void prologue_qk(const PrologueArgs &pro, int s, int n, int h, int sub,
                                            int l8, float (&out)[D / 8]) {
    constexpr int kVec = D / 32;  // slices of 32 channels
    const size_t HD = (size_t)pro.H * D;
    float mine[4] = {0.f, 0.f, 0.f, 0.f};
    float ss = 0.f;
    if (sub < kVec) {
        const int c = 32 * sub + 4 * l8;
        const float *st = pro.conv + ((size_t)n * 3 + s) * 3 * HD + (size_t)h * D + c;
        const float *w = pro.w[s] + ((size_t)h * D + c) * 4;
        float s0[4], s1[4], s2[4], xc[4];
        load4(st, 0, s0);
        load4(st, HD, s1);
        load4(st, 2 * HD, s2);
        load4(static_cast<const Tin *>(pro.x[s]), ((size_t)n * pro.H + h) * D + c, xc);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 t = *reinterpret_cast<const float4 *>(w + 4 * e);
            float cv = t.w * xc[e];
            cv = fmaf(t.z, s2[e], cv);
            cv = fmaf(t.y, s1[e], cv);
            cv = fmaf(t.x, s0[e], cv);
            mine[e] = swish(cv, sizeof(Tin) == 2);
            ss = fmaf(mine[e], mine[e], ss);
        }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float t = ss + pro.l2_eps;
    const float r = t > 0.f ? rsqrtf(t) : 0.f;
#pragma unroll
    for (int i = 0; i < kVec; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            out[4 * i + e] = r * __shfl_sync(0xffffffffu, mine[e], 8 * i + l8);
}

// v of pair (n, h) on value channel `row`
template <int D, typename Tin>
__device__ __forceinline__ float prologue_v(const PrologueArgs &pro, int n, int h, int row) {
    const size_t HD = (size_t)pro.H * D;
    const float *st = pro.conv + ((size_t)n * 3 + 2) * 3 * HD + (size_t)h * D + row;
    const float4 t = *reinterpret_cast<const float4 *>(pro.w[2] + ((size_t)h * D + row) * 4);
    float cv = t.w * to_f(static_cast<const Tin *>(pro.x[2])[((size_t)n * pro.H + h) * D + row]);
    cv = fmaf(t.z, st[2 * HD], cv);
    cv = fmaf(t.y, st[HD], cv);
    cv = fmaf(t.x, st[0], cv);
    return swish(cv, sizeof(Tin) == 2);
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
template <int D, typename Tin, bool kPro>
__global__ void __launch_bounds__(128) decode_step_gated_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
    const float *__restrict__ log_alpha, const float *__restrict__ beta,
    float *__restrict__ S, Tin *__restrict__ y, int NH, const Tin *__restrict__ gate,
    const float *__restrict__ norm_w, float eps, const __grid_constant__ PrologueArgs pro) {
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
    int pn = 0, ph = 0;  // the pair's session and head (prologue)
    if constexpr (kPro) {
        pn = p / pro.H;
        ph = p % pro.H;
        prologue_qk<D, Tin>(pro, 0, pn, ph, sub, l8, qq);
        prologue_qk<D, Tin>(pro, 1, pn, ph, sub, l8, kk);
    }
    // v of the warp's rows (D / 4 of them), one per lane, handed out by shuffles
    const float vlane = kPro && lane < kRowsPerWarp
                            ? prologue_v<D, Tin>(pro, pn, ph, warp * kRowsPerWarp + lane) : 0.f;
#pragma unroll
    for (int i4 = 0; i4 < kVec; ++i4)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 32 * i4 + 4 * l8 + e;
            if constexpr (!kPro) {
                kk[4 * i4 + e] = to_f(k[vec + c]);
                qq[4 * i4 + e] = to_f(q[vec + c]);
            }
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
        const float vr = kPro ? __shfl_sync(0xffffffffu, vlane, row - warp * kRowsPerWarp)
                              : to_f(v[vec + row]);
        const float u = b * (vr - rk);
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
        if constexpr (kPro) {
            // every warp has read the pair's conv state: move it on by one
            // token, (x_{t-2}, x_{t-1}, x_t) per stream
            const size_t HD = (size_t)pro.H * D;
#pragma unroll
            for (int s3 = 0; s3 < 3; ++s3) {
                const int c = 4 * lane;
                if (c < D) {
                    float *st = pro.conv + ((size_t)pn * 3 + s3) * 3 * HD + (size_t)ph * D + c;
                    const float4 a1 = *reinterpret_cast<const float4 *>(st + HD);
                    const float4 a2 = *reinterpret_cast<const float4 *>(st + 2 * HD);
                    float xc[4];
                    load4(static_cast<const Tin *>(pro.x[s3]), ((size_t)pn * pro.H + ph) * D + c, xc);
                    *reinterpret_cast<float4 *>(st) = a1;
                    *reinterpret_cast<float4 *>(st + HD) = a2;
                    *reinterpret_cast<float4 *>(st + 2 * HD) = make_float4(xc[0], xc[1], xc[2], xc[3]);
                }
            }
        }
        __syncwarp();  // all lanes have read the buffer
        if (lane == 0) {
            __threadfence_block();
            atomicAdd(&released[bf], 1);
        }
    }
  }
}

template <int D, typename Tin, bool kGated, bool kPro = false>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *la,
                         const float *beta, float *S, int NH, void *o, cudaStream_t s,
                         const void *gate, const float *norm_w, float eps,
                         const PrologueArgs &pro = PrologueArgs{}) {
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
                             &per, decode_step_gated_kernel<D, Tin, kPro>, 128, 0)
                       : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                             &per, decode_step_kernel<D, Tin>, 128, 0);
        if (e != cudaSuccess) return e;
        res = sms * (per > 0 ? per : 1);
        resident[dev].store(res, std::memory_order_relaxed);
    }
    // as many pairs per block as the resident blocks need, spread evenly:
    // k = ceil(NH / res) pairs per block on ceil(NH / k) blocks
    const int per_block = (NH + res - 1) / res;
    const int grid = (NH + per_block - 1) / per_block;
    if constexpr (kGated)
        decode_step_gated_kernel<D, Tin, kPro><<<grid, 128, 0, s>>>(
            static_cast<const Tin *>(q), static_cast<const Tin *>(k),
                                  static_cast<const Tin *>(v), la, beta, S, static_cast<Tin *>(o),
                                  NH, static_cast<const Tin *>(gate), norm_w, eps, pro);
    else
        decode_step_kernel<D, Tin><<<grid, 128, 0, s>>>(
            static_cast<const Tin *>(q), static_cast<const Tin *>(k),
            static_cast<const Tin *>(v), la, beta, S, static_cast<Tin *>(o), NH);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_layer(const void *const x[3], const float *const w[3], float *conv,
                                float l2_eps, const float *log_alpha, const float *beta,
                                float *S, int N, int H, int d, kda_dtype_t dt, const void *gate,
                                const float *norm_w, float eps, void *y, cudaStream_t s) {
    const int NH = N * H;
    if (NH == 0) return cudaSuccess;
    PrologueArgs pro{};
    for (int i = 0; i < 3; ++i) {
        pro.x[i] = x[i];
        pro.w[i] = w[i];
    }
    pro.conv = conv;
    pro.H = H;
    pro.l2_eps = l2_eps;
    if (d == 128)
        return dt == KDA_BF16
                   ? launch_typed<128, __nv_bfloat16, true, true>(nullptr, nullptr, nullptr, log_alpha,
                                                                  beta, S, NH, y, s, gate, norm_w, eps, pro)
                   : launch_typed<128, float, true, true>(nullptr, nullptr, nullptr, log_alpha, beta,
                                                          S, NH, y, s, gate, norm_w, eps, pro);
    return dt == KDA_BF16
               ? launch_typed<64, __nv_bfloat16, true, true>(nullptr, nullptr, nullptr, log_alpha, beta,
                                                             S, NH, y, s, gate, norm_w, eps, pro)
               : launch_typed<64, float, true, true>(nullptr, nullptr, nullptr, log_alpha, beta, S,
                                                     NH, y, s, gate, norm_w, eps, pro);
}

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

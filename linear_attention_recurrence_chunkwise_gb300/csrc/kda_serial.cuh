// Token-serial KDA steps on CUDA cores, for 64-token chunks whose cumulative
// log-decay leaves the range of the chunk form.
//
// The chunk form factors the decay between two tokens of a chunk onto both of
// them (Gamma on the later token, 1/Gamma on the earlier one, "Kimi Delta
// Attention 完全拆解", chunkwise section), so it needs exp(-G) to stay finite in
// fp32: |G| <= 80 over the chunk.  K3 bounds the per-token log-decay at -5
// ("Kimi K3 的 KDA" section 6), which allows -320 over 64 tokens.  Such
// chunks are taken here one token at a time with the recurrence itself
// ("Kimi Delta Attention 完全拆解", the per-token decode order):
//
//   S <- Diag(alpha_t) S;  u = beta_t (v_t - S^T k_t);  S <- S + k_t u^T;  o_t = S^T q_t
//
// which only multiplies by alpha <= 1 and so holds for any gate, down to
// alpha = 0.  All arithmetic is fp32.
//
// 256 threads take part.  Thread t owns value column v = t % D and the key
// channels c0 .. c0 + kCP - 1 of it (c0 = kCP * (t / D)): kCP = 64 for D = 128
// (two parts per column), 16 for D = 64 (four parts).  The two column sums of
// a token (S^T k and S^T q) add the parts' partial sums through shared memory,
// every part in the same order, so every part computes the same u.
#pragma once

#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {

template <int D>
struct Serial {
    static constexpr int kThreads = 256;
    static constexpr int kParts = kThreads / D;  // threads per value column
    static constexpr int kCP = D / kParts;       // key channels per thread
    static_assert(kParts * kCP == D && kThreads % D == 0, "D must divide 256");
};

__device__ __forceinline__ void serial_store(float *p, float x) { *p = x; }
__device__ __forceinline__ void serial_store(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
}

// bar.sync over the first `count` threads of the block (count a multiple of 32)
__device__ __forceinline__ void serial_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// (a0, a1) *= (b0, b1) and (c0, c1) += (a0, a1) * (b0, b1): packed fp32, round
// to nearest (the same results as the scalar instructions)
__device__ __forceinline__ void serial_mul2(float &a0, float &a1, float b0, float b1) {
    asm("{\n\t.reg .b64 x, y;\n\t"
        "mov.b64 x, {%0, %1};\n\t"
        "mov.b64 y, {%2, %3};\n\t"
        "mul.rn.f32x2 x, x, y;\n\t"
        "mov.b64 {%0, %1}, x;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}
__device__ __forceinline__ void serial_fma2(float &c0, float &c1, float a0, float a1, float b0,
                                            float b1) {
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %5};\n\t"
        "mov.b64 z, {%0, %1};\n\t"
        "fma.rn.f32x2 z, x, y, z;\n\t"
        "mov.b64 {%0, %1}, z;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Four consecutive floats of a staged row (16-byte loads when kVec4: the row
// stride and the thread's first channel are multiples of 4 floats and the rows
// start on 16 bytes).
template <bool kVec4>
__device__ __forceinline__ float4 serial_ld4(const float *p) {
    if constexpr (kVec4) return *reinterpret_cast<const float4 *>(p);
    return make_float4(p[0], p[1], p[2], p[3]);
}

// ntok tokens, staged in shared memory as fp32 rows of stride ld: K, Q, A
// (alpha itself, not its log) [ntok][ld] over key channels, V [ntok][ld] over
// value channels, bet [ntok].  s holds this thread's state entries S[c0 + i][v].
// Threads 0 .. 255 call this together; bar_id names the barrier they use.
//
// Column sums go through red_r, float[2][kParts][D] (double-buffered by token
// parity, so one barrier per token orders both its writes and the next
// token's).  Outputs:
//  - kDeferO: token r's per-part partial sums of o are left in
//    red_o[(r * kParts + part) * D + v] (red_o: float[ntok][kParts][D]); the
//    caller adds the parts after a barrier.
//  - otherwise: o[o_base + r * o_stride + v] is stored here, unless o is null
//    (a second barrier per token; n_o is o's extent, for the bounds-checked
//    build).
template <int D, bool kVec4, bool kDeferO, typename Tout>
__device__ __forceinline__ void serial_tokens(float (&s)[Serial<D>::kCP], const float *K,
                                              const float *Q, const float *A, const float *V,
                                              const float *bet, int ld, int ntok, float *red_r,
                                              float *red_o, Tout *o, size_t o_base,
                                              size_t o_stride, size_t n_o, int32_t *status,
                                              int bar_id) {
    constexpr int P = Serial<D>::kParts, CP = Serial<D>::kCP;
    static_assert(CP % 4 == 0, "four channels per load");
    const int t = threadIdx.x, v = t % D, part = t / D, c0 = part * CP;
    for (int r = 0; r < ntok; ++r) {
        const float *kr = K + (size_t)r * ld + c0;
        const float *qr = Q + (size_t)r * ld + c0;
        const float *ar = A + (size_t)r * ld + c0;
        float *rr = red_r + (r & 1) * P * D;
        // decay, then this part's share of (S^T k)_v in two packed sums
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < CP; i += 4) {
            const float4 a4 = serial_ld4<kVec4>(ar + i), k4 = serial_ld4<kVec4>(kr + i);
            serial_mul2(s[i], s[i + 1], a4.x, a4.y);
            serial_mul2(s[i + 2], s[i + 3], a4.z, a4.w);
            serial_fma2(acc[0], acc[1], s[i], s[i + 1], k4.x, k4.y);
            serial_fma2(acc[2], acc[3], s[i + 2], s[i + 3], k4.z, k4.w);
        }
        rr[part * D + v] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        serial_bar(bar_id, Serial<D>::kThreads);
        float sk = 0.f;
#pragma unroll
        for (int j = 0; j < P; ++j) sk += rr[j * D + v];
        const float u = bet[r] * (V[(size_t)r * ld + v] - sk);
        // rank-one write, then this part's share of (S^T q)_v
        float oc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < CP; i += 4) {
            const float4 k4 = serial_ld4<kVec4>(kr + i), q4 = serial_ld4<kVec4>(qr + i);
            serial_fma2(s[i], s[i + 1], k4.x, k4.y, u, u);
            serial_fma2(s[i + 2], s[i + 3], k4.z, k4.w, u, u);
            serial_fma2(oc[0], oc[1], s[i], s[i + 1], q4.x, q4.y);
            serial_fma2(oc[2], oc[3], s[i + 2], s[i + 3], q4.z, q4.w);
        }
        const float op = (oc[0] + oc[1]) + (oc[2] + oc[3]);
        if constexpr (kDeferO) {
            red_o[((size_t)r * P + part) * D + v] = op;
        } else {
            red_o[part * D + v] = op;
            serial_bar(bar_id, Serial<D>::kThreads);
            if (part == 0 && o) {
                float ov = 0.f;
#pragma unroll
                for (int j = 0; j < P; ++j) ov += red_o[j * D + v];
                const size_t oi = o_base + (size_t)r * o_stride + v;
                if (in_bounds(status, oi, n_o)) serial_store(o + oi, ov);
            }
        }
    }
}

}  // namespace kda

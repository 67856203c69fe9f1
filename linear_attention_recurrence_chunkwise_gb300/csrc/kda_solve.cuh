// T' = (I + A)^-1 diag(beta) for a 64 x 64 strictly lower-triangular A -- the
// UT/WY solve of a 64-token chunk -- on the warp-level tensor cores (mma.sync,
// TF32 inputs, fp32 accumulate), written in bf16 as the 128-byte-swizzled
// operand tile of the W and U~ products.
//
// With T = (I + A)^-1 cut into 16 x 16 blocks T_IJ (I >= J):
//   1. the diagonal blocks T_II, by forward substitution (one lane per column);
//   2. T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32 T_22 (one warp each), which
//      completes the two 32 x 32 diagonal halves of T;
//   3. the lower-left 32 x 32 half, T_IJ = -sum_K T_IK X_KJ with
//      X_KJ = sum_L A_KL T_LJ (I, K in {2, 3}; J, L in {0, 1}), one warp per
//      output block.
// Each warp keeps the intermediate X in mma.sync accumulator registers and
// feeds it straight into the next product as its B operand (see mma_xt and
// mma_tx), so a chain of block products never goes through shared memory.
// Three dependent steps with two barriers in between, instead of one step per
// block diagonal.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_sm100.cuh"

namespace kda {

constexpr int kSolveLd = 68;  // fp32 row stride of the matrix

// d (16 x 8, fp32) += a (16 x 8, tf32) * b (8 x 8, tf32).  The operands are
// passed as fp32 bit patterns: the tensor cores read their tf32 part (the low
// 13 mantissa bits are dropped), which spares a conversion per operand.
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4],
                                                const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// p += (A_KL T_LJ)^T as two m16n8 accumulator fragments (p[nt] = columns
// 8 nt .. 8 nt + 7 of the transpose).  tl -> 16 x 16 block T_LJ, ak -> A_KL,
// both fp32 with row stride kSolveLd.  The transpose is what lets mma_tx use
// the result as a B operand without leaving registers.
__device__ __forceinline__ void mma_xt(float (&p)[2][4], const float *tl, const float *ak,
                                       int lane) {
    const int g = lane >> 2, t = lane & 3;
    constexpr int ld = kSolveLd;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4];  // A operand = T_LJ^T: element (m, k) = T_LJ[k][m]
        a[0] = __float_as_uint(tl[(8 * ks + t) * ld + g]);
        a[1] = __float_as_uint(tl[(8 * ks + t) * ld + g + 8]);
        a[2] = __float_as_uint(tl[(8 * ks + t + 4) * ld + g]);
        a[3] = __float_as_uint(tl[(8 * ks + t + 4) * ld + g + 8]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {  // B operand = A_KL^T: (k, n) = A_KL[n][k]
            uint32_t b[2];
            b[0] = __float_as_uint(ak[(8 * nt + g) * ld + 8 * ks + t]);
            b[1] = __float_as_uint(ak[(8 * nt + g) * ld + 8 * ks + t + 4]);
            mma_tf32_16x8x8(p[nt], a, b);
        }
    }
}

// z += T_IK X_KJ with X_KJ^T held in the accumulator fragments p (from
// mma_xt).  An accumulator fragment gives lane (g, t) the entries
// X[8 ks + 2t][n] and X[8 ks + 2t + 1][n] for n = g and g + 8, which is a B
// fragment once the eight k of each step are taken in the order 2t, 2t + 1
// instead of t, t + 4; the A fragment of T_IK is loaded in that same order, so
// the sum over k is unchanged.
__device__ __forceinline__ void mma_tx(float (&z)[2][4], const float *tk, const float (&p)[2][4],
                                       int lane) {
    const int g = lane >> 2, t = lane & 3;
    constexpr int ld = kSolveLd;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const float2 r0 = *reinterpret_cast<const float2 *>(tk + g * ld + 8 * ks + 2 * t);
        const float2 r1 = *reinterpret_cast<const float2 *>(tk + (g + 8) * ld + 8 * ks + 2 * t);
        uint32_t a[4];  // T_IK
        a[0] = __float_as_uint(r0.x);
        a[1] = __float_as_uint(r1.x);
        a[2] = __float_as_uint(r0.y);
        a[3] = __float_as_uint(r1.y);
#pragma unroll
        for (int nz = 0; nz < 2; ++nz) {
            uint32_t b[2];
            b[0] = __float_as_uint(p[ks][2 * nz]);
            b[1] = __float_as_uint(p[ks][2 * nz + 1]);
            mma_tf32_16x8x8(z[nz], a, b);
        }
    }
}

// Block (I, J) of T, I >= J: the diagonal blocks sit in place, a lower block
// T_IJ in the upper-triangle slot (J, I), which A leaves free.
__device__ __forceinline__ float *t_block(float *as, int bi, int bj) {
    return as + (16 * bj) * kSolveLd + 16 * bi;
}
__device__ __forceinline__ const float *a_block(const float *as, int bi, int bj) {
    return as + (16 * bi) * kSolveLd + 16 * bj;
}

// Byte offset of bf16 element (row, col) of a 64 x 64 tile with 128-byte rows
// and the 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t tp_offset(int row, int col) {
    return (row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 3) ^ row) & 7) << 4) + (col & 7) * 2;
}

// T'_IJ = -z diag(beta) (z from mma_tx) into the bf16 tile.
__device__ __forceinline__ void store_tprime(uint8_t *tp, const float *beta, int bi, int bj,
                                             const float (&z)[2][4], int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nz = 0; nz < 2; ++nz) {
        const int col = 16 * bj + 8 * nz + 2 * t;
        const float b0 = beta[col], b1 = beta[col + 1];
        *reinterpret_cast<uint32_t *>(tp + tp_offset(16 * bi + g, col)) =
            sm100::pack_bf16(-z[nz][0] * b0, -z[nz][1] * b1);
        *reinterpret_cast<uint32_t *>(tp + tp_offset(16 * bi + g + 8, col)) =
            sm100::pack_bf16(-z[nz][2] * b0, -z[nz][3] * b1);
    }
}

// On entry `as` (fp32, row stride kSolveLd) holds A strictly below the
// diagonal (what lies on and above it is never read), and beta[64] (16-byte
// aligned) the token weights.  The blocks of T it writes back for later steps
// are fp32 too, read by the tensor cores at tf32 precision (the forward
// substitution of step 1 uses A in full).  On exit `tp` holds T' (bf16, [r][j], 128-byte
// swizzle) and `as` is scratch.  Called by the 128 threads (pt = 0 .. 127) of
// four warps, which synchronise among themselves on the named barrier `bar`.
// The caller makes the tile visible to the tensor cores (fence.proxy.async)
// and synchronises the four warps.  kOffloadDiag moves the bf16 stores of the
// diagonal blocks of T' from the substituting warps (0, 1) of step 1 to the
// idle warps (2, 3) of step 2, which read T_bb back: faster when every SM of
// the GPU is busy, slower otherwise.
template <bool kOffloadDiag>
__device__ __forceinline__ void solve_tprime64(float *as, const float *beta, uint8_t *tp, int pt,
                                               uint32_t bar) {
    constexpr int ld = kSolveLd;
    const int warp = pt >> 5, lane = pt & 31;
    // zero the six blocks above the diagonal of T' (96 pieces: 16 rows x 16
    // bytes of each block), from the threads that have no column in step 1
    for (int q = pt - 64; q >= 0 && q < 96; q += 64) {
        const int blk = q >> 4, piece = q & 15;
        const int bi = blk < 3 ? 0 : blk < 5 ? 1 : 2;
        const int bj = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
        const int row = 16 * bi + piece;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            *reinterpret_cast<uint4 *>(tp + tp_offset(row, 16 * bj + 8 * h)) =
                make_uint4(0, 0, 0, 0);
    }
    // 1. diagonal blocks: lane = column c of block b, substitution down the
    //    rows, each row's sum taken over i = 0, 1, ... in order
    if (pt < 64) {
        const int b = pt >> 4, c = pt & 15;
        float *Ab = as + (16 * b) * ld + 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = r == c ? 1.f : 0.f;
#pragma unroll
        for (int i4 = 0; i4 < 16; i4 += 4) {
            float4 a[16];  // A[r][i4 .. i4 + 3] for the rows still to update
#pragma unroll
            for (int r = i4 + 1; r < 16; ++r)
                a[r] = *reinterpret_cast<const float4 *>(Ab + r * ld + i4);
#pragma unroll
            for (int i = i4; i < i4 + 4; ++i) {
#pragma unroll
                for (int r = i + 1; r < 16; ++r) {
                    const float4 v = a[r];
                    const float air = i - i4 == 0 ? v.x : i - i4 == 1 ? v.y : i - i4 == 2 ? v.z : v.w;
                    x[r] = fmaf(-air, x[i], x[r]);
                }
            }
        }
        __syncwarp();
        // T_bb is read back as a tensor-core operand (and, with kOffloadDiag,
        // by warps 2 and 3 for its bf16 copy in T')
#pragma unroll
        for (int r = 0; r < 16; ++r)
            Ab[r * ld + c] = x[r];
        if constexpr (!kOffloadDiag) {
            const float bc = beta[16 * b + c];
#pragma unroll
            for (int r = 0; r < 16; ++r)
                *reinterpret_cast<__nv_bfloat16 *>(tp + tp_offset(16 * b + r, 16 * b + c)) =
                    __float2bfloat16_rn(x[r] * bc);
        }
    }
    sm100::named_bar_sync(bar, 128);
    // 2. T_10 (warp 0) and T_32 (warp 1); with kOffloadDiag, warps 2 and 3
    //    meanwhile write the diagonal blocks of T' = T diag(beta) in bf16 from
    //    T_bb, 8 columns of a row per piece, two pieces per thread
    if constexpr (kOffloadDiag) {
        if (warp >= 2) {
#pragma unroll
            for (int q = pt - 64; q < 128; q += 64) {
                const int b = q >> 5, r = (q >> 1) & 15, h = q & 1;
                const float *src = as + (16 * b + r) * ld + 16 * b + 8 * h;
                const float4 t0 = *reinterpret_cast<const float4 *>(src);
                const float4 t1 = *reinterpret_cast<const float4 *>(src + 4);
                const float4 b0 = *reinterpret_cast<const float4 *>(beta + 16 * b + 8 * h);
                const float4 b1 = *reinterpret_cast<const float4 *>(beta + 16 * b + 8 * h + 4);
                uint4 w;
                w.x = sm100::pack_bf16(t0.x * b0.x, t0.y * b0.y);
                w.y = sm100::pack_bf16(t0.z * b0.z, t0.w * b0.w);
                w.z = sm100::pack_bf16(t1.x * b1.x, t1.y * b1.y);
                w.w = sm100::pack_bf16(t1.z * b1.z, t1.w * b1.w);
                *reinterpret_cast<uint4 *>(tp + tp_offset(16 * b + r, 16 * b + 8 * h)) = w;
            }
        }
    }
    if (warp < 2) {
        const int bi = 2 * warp + 1, bj = 2 * warp;
        float p[2][4] = {}, z[2][4] = {};
        mma_xt(p, t_block(as, bj, bj), a_block(as, bi, bj), lane);
        mma_tx(z, t_block(as, bi, bi), p, lane);
        const int g = lane >> 2, t = lane & 3;
        float *dst = t_block(as, bi, bj);
#pragma unroll
        for (int nz = 0; nz < 2; ++nz) {
            // (read back only as a tensor-core operand)
            *reinterpret_cast<float2 *>(dst + g * ld + 8 * nz + 2 * t) =
                make_float2(-z[nz][0], -z[nz][1]);
            *reinterpret_cast<float2 *>(dst + (g + 8) * ld + 8 * nz + 2 * t) =
                make_float2(-z[nz][2], -z[nz][3]);
        }
        store_tprime(tp, beta, bi, bj, z, lane);
    }
    sm100::named_bar_sync(bar, 128);
    // 3. T_IJ, (I, J) = (2, 0), (2, 1), (3, 0), (3, 1) for warps 0 .. 3
    {
        const int bj = warp & 1, bi = 2 + (warp >> 1);
        float p2[2][4] = {}, z[2][4] = {};
        // X_2J = sum_{L = J}^{1} A_2L T_LJ
        if (bj == 0) mma_xt(p2, t_block(as, 0, 0), a_block(as, 2, 0), lane);
        mma_xt(p2, t_block(as, 1, bj), a_block(as, 2, 1), lane);
        if (bi == 2) {
            mma_tx(z, t_block(as, 2, 2), p2, lane);
        } else {
            float p3[2][4] = {};  // X_3J
            if (bj == 0) mma_xt(p3, t_block(as, 0, 0), a_block(as, 3, 0), lane);
            mma_xt(p3, t_block(as, 1, bj), a_block(as, 3, 1), lane);
            mma_tx(z, t_block(as, 3, 2), p2, lane);
            mma_tx(z, t_block(as, 3, 3), p3, lane);
        }
        store_tprime(tp, beta, bi, bj, z, lane);
    }
}

}  // namespace kda

// Inverse of a 64 x 64 unit lower-triangular matrix, (I + A)^-1 with A
// strictly lower, on the warp-level tensor cores (mma.sync, TF32 inputs, fp32
// accumulate) -- the UT/WY solve of a 64-token chunk.
//
// Layout: fp32 row-major with row stride kSolveLd.  On entry `as` holds A
// (zero on and above the diagonal).  The diagonal 16 x 16 blocks are inverted
// by forward substitution (one lane per column); the off-diagonal blocks then
// follow diagonal by diagonal, T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj, as
// 16 x 16 x 16 mma.sync products.  On exit T_ii sits in the diagonal block and
// T_ij (i > j) in the otherwise unused upper block (j, i); inv_entry() reads T.
// Every block product reads its operands from shared memory once, so the
// solve costs a few hundred shared-memory cycles instead of thousands.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_sm100.cuh"

namespace kda {

constexpr int kSolveLd = 68;     // fp32 row stride of the matrix
constexpr int kSolveYLd = 20;    // fp32 row stride of a 16 x 16 scratch block

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// d (16 x 8, fp32) += a (16 x 8, tf32) * b (8 x 8, tf32)
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4],
                                                const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc[nt] += X (16 x 16 block at xs, row stride ldx) * Y (16 x 16 block at ys,
// row stride ldy), the two 8-column halves of the product in acc[0], acc[1]
// (mma.sync accumulator fragments).
__device__ __forceinline__ void mma_block16(float (&acc)[2][4], const float *xs, int ldx,
                                            const float *ys, int ldy, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        uint32_t a[4];
        a[0] = to_tf32(xs[g * ldx + 8 * ks + t]);
        a[1] = to_tf32(xs[(g + 8) * ldx + 8 * ks + t]);
        a[2] = to_tf32(xs[g * ldx + 8 * ks + t + 4]);
        a[3] = to_tf32(xs[(g + 8) * ldx + 8 * ks + t + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t b[2];
            b[0] = to_tf32(ys[(8 * ks + t) * ldy + 8 * nt + g]);
            b[1] = to_tf32(ys[(8 * ks + t + 4) * ldy + 8 * nt + g]);
            mma_tf32_16x8x8(acc[nt], a, b);
        }
    }
}

// Store scale * acc (16 x 16 accumulator fragments) into a row-major block.
__device__ __forceinline__ void store_block16(float *dst, int ld, const float (&acc)[2][4],
                                              float scale, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2 *>(dst + g * ld + 8 * nt + 2 * t) =
            make_float2(scale * acc[nt][0], scale * acc[nt][1]);
        *reinterpret_cast<float2 *>(dst + (g + 8) * ld + 8 * nt + 2 * t) =
            make_float2(scale * acc[nt][2], scale * acc[nt][3]);
    }
}

// Block (bi, bj) of T lives at row 16 bj, column 16 bi for bi >= bj (the
// diagonal blocks in place, the lower blocks mirrored into the upper half).
__device__ __forceinline__ const float *t_block(const float *as, int bi, int bj) {
    return as + (16 * bj) * kSolveLd + 16 * bi;
}

// Byte offset of bf16 element (row, col) of a 64 x 64 tile with 128-byte rows
// and the 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t tp_offset(int row, int col) {
    return (row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 3) ^ row) & 7) << 4) + (col & 7) * 2;
}

// Optional second output of the inverse: T' = T diag(beta) in bf16, written
// straight from the registers that produce T into a swizzled tile (the B
// operand of the W and U~ products).
struct TprimeOut {
    uint8_t *tile;      // 64 x 64 bf16, 128-byte swizzle; nullptr: no second output
    const float *beta;  // column scale, 64 values
};

// T = (I + A)^-1 in place in `as` (see the file comment), and T' when
// `out.tile` is set.  `ys` is scratch for three 16 x kSolveYLd blocks.  Called
// by 256 threads (8 warps) that all reach the named barrier `bar` (id)
// between the stages.
__device__ __forceinline__ void inverse_unit_lower64(float *as, float *ys, int pt, uint32_t bar,
                                                     TprimeOut out = {nullptr, nullptr}) {
    const int warp = pt >> 5, lane = pt & 31;
    // diagonal 16 x 16 blocks: lane = column c of block b, forward substitution
    if (pt < 64) {
        const int b = pt >> 4, c = pt & 15;
        float *Ab = as + (16 * b) * kSolveLd + 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = r == c ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < r; i += 4) {  // A is zero on and above the diagonal
                const float4 a = *reinterpret_cast<const float4 *>(Ab + r * kSolveLd + i);
                acc = fmaf(-a.x, x[i], acc);
                acc = fmaf(-a.y, x[i + 1], acc);
                acc = fmaf(-a.z, x[i + 2], acc);
                acc = fmaf(-a.w, x[i + 3], acc);
            }
            x[r] = acc;
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 16; ++r) Ab[r * kSolveLd + c] = x[r];
        if (out.tile) {
            const float bc = out.beta[16 * b + c];
#pragma unroll
            for (int r = 0; r < 16; ++r)
                *reinterpret_cast<__nv_bfloat16 *>(out.tile + tp_offset(16 * b + r, 16 * b + c)) =
                    __float2bfloat16_rn(x[r] * bc);
        }
    } else if (out.tile && pt < 64 + 96) {
        // zero the six blocks above the diagonal of T' (16-byte pieces)
        const int q = pt - 64, blk = q >> 4, piece = q & 15;  // 6 blocks x 16 rows
        const int bi = blk < 3 ? 0 : blk < 5 ? 1 : 2;
        const int bj = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
        const int row = 16 * bi + piece;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            *reinterpret_cast<uint4 *>(out.tile + tp_offset(row, 16 * bj + 8 * h)) =
                make_uint4(0, 0, 0, 0);
    }
    sm100::named_bar_sync(bar, 256);
    // off-diagonal blocks, one block per warp, diagonal d = 1, 2, 3
#pragma unroll
    for (int d = 1; d < 4; ++d) {
        if (warp < 4 - d) {
            const int bi = warp + d, bj = warp;
            float *Y = ys + warp * 16 * kSolveYLd;
            float acc[2][4] = {};
            for (int k = bj; k < bi; ++k)  // Y = sum_k A_ik T_kj
                mma_block16(acc, as + (16 * bi) * kSolveLd + 16 * k, kSolveLd,
                            t_block(as, k, bj), kSolveLd, lane);
            store_block16(Y, kSolveYLd, acc, 1.f, lane);
            __syncwarp();
            float tt[2][4] = {};
            mma_block16(tt, t_block(as, bi, bi), kSolveLd, Y, kSolveYLd, lane);
            store_block16(as + (16 * bj) * kSolveLd + 16 * bi, kSolveLd, tt, -1.f, lane);
            if (out.tile) {  // T' block (bi, bj) = -tt scaled by beta along columns
                const int g = lane >> 2, t = lane & 3;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int col = 16 * bj + 8 * nt + 2 * t;
                    const float b0 = out.beta[col], b1 = out.beta[col + 1];
                    *reinterpret_cast<uint32_t *>(out.tile + tp_offset(16 * bi + g, col)) =
                        sm100::pack_bf16(-tt[nt][0] * b0, -tt[nt][1] * b1);
                    *reinterpret_cast<uint32_t *>(out.tile + tp_offset(16 * bi + g + 8, col)) =
                        sm100::pack_bf16(-tt[nt][2] * b0, -tt[nt][3] * b1);
                }
            }
        }
        sm100::named_bar_sync(bar, 256);
    }
}

// Entry (r, j) of T after inverse_unit_lower64.
__device__ __forceinline__ float inv_entry(const float *as, int r, int j) {
    if (j > r) return 0.f;
    const int bi = r >> 4, bj = j >> 4;
    return t_block(as, bi, bj)[(r & 15) * kSolveLd + (j & 15)];
}

}  // namespace kda

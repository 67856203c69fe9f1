// Tensor-core chunkwise KDA forward for sm_103a (bf16 q/k/v, d_k = d_v = 128).
//
// One CTA per (sequence, head) walks the sequence in 64-token chunks.  The
// algorithm is the chunk form of the recurrence (see the CUDA-core engine for
// the derivation; "Kimi Delta Attention 完全拆解", chunkwise section; "Kimi K3
// 的 KDA" section 5):
//
//   G = in-chunk inclusive cumsum of log_alpha, Gamma = exp(G), gamma = Gamma_last
//   Kh = K . Gamma,  Qh = Q . Gamma,  Kb = K / Gamma                       (a1, a2)
//   R  = [Kh; Qh] Kb^T            A = StrictTril(diag(beta) R_top)          (a3)
//   T' = (I + A)^-1 diag(beta)    W = T' Kh,  U~ = T' V                     (a4)
//   M  = Tril(R_bottom)                                                    (a5)
//   U  = U~ - W S,   O = Qh S + M U,   S <- Diag(gamma) (S + Kb^T U)       (a6)
//
// Every contraction runs on tcgen05 with M = 128 by working in the transposed
// frame: the feature axis (d_k or d_v = 128) is the MMA's M dimension and
// tokens are N or K.  So the products are U^T = U~^T - S^T W^T, O^T = S^T Qh^T
// + U^T M^T, (S^T)' = S^T + U^T Kb, W^T = Kh^T T'^T, U~^T = V^T T'^T, and R
// stacks Kh and Qh as the 128 rows of one A operand.  The fp32 state lives in
// tensor memory for the whole sequence (the S-update MMA accumulates into it);
// a bf16 copy in shared memory is the MMA operand.
//
// Warp roles (288 threads):
//   warp 0      TMA producer: q, k, v tiles (64 tokens x 64 channels, 128-byte
//               swizzle) into a two-stage ring; allocates tensor memory.
//   warps 1-4   chunk-local work for chunk n+1 (a1-a5): gates, scaled operands,
//               R, masks, the triangular solve, W and U~.
//   warps 5-8   the serial carry for chunk n (a6) and the output store.
// The chunk-local work of the next chunk overlaps the carry of the current one.
//
// Every wait is bounded in time; on a timeout the kernel records
// KDA_ERR_TIMEOUT, runs its remaining steps without waiting, drains its own
// copies and MMAs, frees tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int D = 128;
constexpr int C = kChunk;
constexpr int kPrepWarp0 = 1;
constexpr int kEpiWarp0 = 5;
constexpr int kThreads = 32 * 9;
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns (fp32 accumulators, 128 lanes each)
constexpr uint32_t kColRW = 0;    // R, then W^T              (64 columns)
constexpr uint32_t kColU = 64;    // U~^T / U^T, two buffers (2 x 64)
constexpr uint32_t kColO = 192;   // O^T, two buffers         (2 x 64)
constexpr uint32_t kColS = 384;   // S^T master copy, fp32    (128)
constexpr int LDA = 68;           // fp32 row stride of the solve matrix
constexpr uint32_t kBarPrep = 1, kBarEpi = 2;  // named barrier ids
constexpr uint32_t kTileBytes = 64 * 64 * 2;   // one TMA box

struct __align__(1024) TcStage {
    uint8_t kq[32768];  // per 64-channel slab: Kh rows 0-63 | Qh rows 0-63; Kh area -> -W
    uint8_t v[16384];   // V [token][v], two slabs
    uint8_t kb[16384];  // Kb [token][c], two slabs
    uint8_t m[8192];    // output mask [r][j]
    float gam[D];       // gamma per key channel
    float bet[C];       // beta per token (0 past the end)
    uint8_t pad[256];
};

struct __align__(1024) TcSmem {
    TcStage st[2];
    uint8_t tp[8192];   // T' bf16 [r][j]; fp32 scratch while solving
    uint8_t ut[16384];  // U^T bf16 [v][j]
    uint8_t sb[32768];  // S^T bf16 [v][c], two slabs
    float as[C * LDA];  // solve matrix / block inverse (fp32)
    uint64_t full[2], ready[2], empty[2], uempty[2];
    uint64_t bar_r, bar_w, bar_u, bar_s, bar_fin;
    uint32_t tmem_base;
    int abort;
    int domain;
};

// Wait for a phase; on timeout (or once any thread has timed out) return
// without waiting so that every thread still reaches every barrier.
__device__ __forceinline__ void wait_phase(uint64_t &bar, uint32_t parity, volatile int *abort) {
    mbar_wait(smem_u32(&bar), parity, abort);
}

// The same, executed by all 32 lanes of a warp, which leave it converged (the
// .sync.aligned tcgen05 instructions that follow need the whole warp).
__device__ __forceinline__ void wait_phase_warp(uint64_t &bar, uint32_t parity,
                                                volatile int *abort) {
    mbar_wait(smem_u32(&bar), parity, abort);
    __syncwarp();
}

__device__ __forceinline__ void wait_drain(uint64_t &bar, uint32_t parity) {
    if (mbar_try_wait(smem_u32(&bar), parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&bar), parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                      pack_bf16(f[6], f[7]));
}

// Store 16 fp32 values (one row segment of 16 consecutive bf16 columns) into a
// 128-byte-swizzled tile at (row, col16 .. col16 + 15).
__device__ __forceinline__ void store_row16(uint8_t *tile, int row, int col16,
                                            const float (&f)[16]) {
    float a[8], b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a[j] = f[j];
        b[j] = f[8 + j];
    }
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, col16)) = pack8(a);
    *reinterpret_cast<uint4 *>(tile + sw128_offset(row, col16 + 8)) = pack8(b);
}

// T' = (I + A)^{-1} diag(beta) for the 64 x 64 strictly lower A in sm.as,
// by 16 x 16 blocks: invert the diagonal blocks by forward substitution, then
// the off-diagonal blocks diagonal by diagonal, T_ij = -T_ii sum_{k=j}^{i-1}
// A_ik T_kj.  T_ij (i > j) is kept in the unused upper block (j, i) of sm.as,
// so T_kj for k >= j always sits at row 16 j + ., column block k.
__device__ __forceinline__ void solve_ut(TcSmem &sm, const float *bet, int pt) {
    float *A = sm.as;
    float *Y = reinterpret_cast<float *>(sm.tp);
    if (pt < 64) {
        const int b = pt >> 4, j = pt & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = r == j ? 1.f : 0.f;
#pragma unroll
        for (int i = 0; i < 15; ++i)
#pragma unroll
            for (int r = i + 1; r < 16; ++r)
                x[r] = fmaf(-A[(16 * b + r) * LDA + 16 * b + i], x[i], x[r]);
        named_bar_sync(kBarPrep, 128);
#pragma unroll
        for (int r = 0; r < 16; ++r) A[(16 * b + r) * LDA + 16 * b + j] = x[r];
    } else {
        named_bar_sync(kBarPrep, 128);
    }
    named_bar_sync(kBarPrep, 128);

    const int r = pt >> 3, c = 2 * (pt & 7);
#pragma unroll
    for (int d = 1; d < 4; ++d) {
        // Y_ij = -sum_{k=j}^{i-1} A_ik T_kj  for every block (i, j = i - d)
        for (int bi = d; bi < 4; ++bi) {
            const int bj = bi - d;
            float y0 = 0.f, y1 = 0.f;
            for (int k = bj; k < bi; ++k) {
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const float a = A[(16 * bi + r) * LDA + 16 * k + kk];
                    const float2 t =
                        *reinterpret_cast<const float2 *>(&A[(16 * bj + kk) * LDA + 16 * k + c]);
                    y0 = fmaf(a, t.x, y0);
                    y1 = fmaf(a, t.y, y1);
                }
            }
            *reinterpret_cast<float2 *>(&Y[(bi - d) * 256 + r * 16 + c]) = make_float2(-y0, -y1);
        }
        named_bar_sync(kBarPrep, 128);
        // T_ij = T_ii Y_ij, stored in the upper block (j, i)
        for (int bi = d; bi < 4; ++bi) {
            const int bj = bi - d;
            float t0 = 0.f, t1 = 0.f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const float a = A[(16 * bi + r) * LDA + 16 * bi + kk];
                const float2 y = *reinterpret_cast<const float2 *>(&Y[(bi - d) * 256 + kk * 16 + c]);
                t0 = fmaf(a, y.x, t0);
                t1 = fmaf(a, y.y, t1);
            }
            *reinterpret_cast<float2 *>(&A[(16 * bj + r) * LDA + 16 * bi + c]) =
                make_float2(t0, t1);
        }
        named_bar_sync(kBarPrep, 128);
    }

    // T'[row][j] = T[row][j] beta_j in bf16, 128-byte swizzled [r][j]
    const int row = pt >> 1, half = pt & 1;
    const int bi = row >> 4;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int j0 = 32 * half + 8 * q;
        const int bj = j0 >> 4;
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int j = j0 + e;
            float t = 0.f;
            if (bj <= bi && j <= row) t = A[(16 * bj + (row & 15)) * LDA + 16 * bi + (j & 15)];
            f[e] = t * bet[j];
        }
        *reinterpret_cast<uint4 *>(sm.tp + sw128_offset(row, j0)) = pack8(f);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smem_raw[];
    TcSmem &sm = *reinterpret_cast<TcSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (*p.status == KDA_ERR_INVALID_ARGUMENT) return;  // set by the schedule kernel

    const int h = blockIdx.x % p.H;
    const int rank = blockIdx.x / p.H;
    const int nseq = p.order ? p.order[rank] : rank;
    int64_t start;
    int len;
    seq_range(p, nseq, start, len);
    const int nchunks = (len + C - 1) / C;
    const size_t state_off = ((size_t)nseq * p.H + h) * D * D;
    if (nchunks == 0) {  // empty sequence: the state passes through
        if (p.S_T)
            for (int i = tid; i < D * D; i += kThreads)
                p.S_T[state_off + i] = p.S0 ? p.S0[state_off + i] : 0.f;
        return;
    }

    volatile int *abort = &sm.abort;
    if (tid == 0) {
        sm.abort = 0;
        sm.domain = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.ready[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 2);
            mbar_init(smem_u32(&sm.uempty[s]), 1);
        }
        mbar_init(smem_u32(&sm.bar_r), 1);
        mbar_init(smem_u32(&sm.bar_w), 1);
        mbar_init(smem_u32(&sm.bar_u), 1);
        mbar_init(smem_u32(&sm.bar_s), 1);
        mbar_init(smem_u32(&sm.bar_fin), 2);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int L = 32 * (warp & 3) + lane;  // this thread's TMEM lane

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            int issued = 0;
            for (int n = 0; n < nchunks; ++n) {
                const int s = n & 1;
                if (n >= 2) wait_phase(sm.empty[s], ((n >> 1) - 1) & 1, abort);
                const uint32_t fb = smem_u32(&sm.full[s]);
                mbar_arrive_expect_tx(fb, 6 * kTileBytes);
                const int t0 = static_cast<int>(start + (int64_t)n * C);
                TcStage &S = sm.st[s];
                tma_load_3d(smem_u32(S.kq), &tm_k, fb, 0, h, t0);
                tma_load_3d(smem_u32(S.kq + 8192), &tm_q, fb, 0, h, t0);
                tma_load_3d(smem_u32(S.kq + 16384), &tm_k, fb, 64, h, t0);
                tma_load_3d(smem_u32(S.kq + 24576), &tm_q, fb, 64, h, t0);
                tma_load_3d(smem_u32(S.v), &tm_v, fb, 0, h, t0);
                tma_load_3d(smem_u32(S.v + 8192), &tm_v, fb, 64, h, t0);
                issued = n + 1;
                if (n + 2 < nchunks) {
                    const int t2 = t0 + 2 * C;
                    tma_prefetch_3d(&tm_k, 0, h, t2);
                    tma_prefetch_3d(&tm_k, 64, h, t2);
                    tma_prefetch_3d(&tm_q, 0, h, t2);
                    tma_prefetch_3d(&tm_q, 64, h, t2);
                    tma_prefetch_3d(&tm_v, 0, h, t2);
                    tma_prefetch_3d(&tm_v, 64, h, t2);
                }
            }
            // never leave with a copy in flight
            for (int n = issued > 2 ? issued - 2 : 0; n < issued; ++n)
                wait_drain(sm.full[n & 1], (n >> 1) & 1);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------ chunk-local work (a1-a5)
        const int pt = tid - 32 * kPrepWarp0;
        const int cg = pt >> 3, tg = pt & 7;  // 8 channels x 8 tokens per thread
        const int c0 = 8 * cg;
        const int slab = c0 >> 6, col = c0 & 63;
        bool domain_ok = true;
        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            TcStage &S = sm.st[s];
            const int64_t t0 = start + (int64_t)n * C;
            const int valid = min(C, len - n * C);

            // a1: in-chunk cumulative log-decay, G[t][c] = sum_{t' <= t} log_alpha
            float g[8][8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = 8 * tg + i;
                if (t < valid) {
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.log_alpha + ((size_t)(t0 + t) * p.H + h) * D + c0);
                    const float4 a = src[0], b = src[1];
                    g[i][0] = a.x; g[i][1] = a.y; g[i][2] = a.z; g[i][3] = a.w;
                    g[i][4] = b.x; g[i][5] = b.y; g[i][6] = b.z; g[i][7] = b.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) g[i][e] = 0.f;
                }
            }
            const float bet = (pt < C && pt < valid) ? p.beta[(size_t)(t0 + pt) * p.H + h] : 0.f;
#pragma unroll
            for (int i = 1; i < 8; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) g[i][e] += g[i - 1][e];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float tot = g[7][e];
                float inc = tot;
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    const float up = __shfl_up_sync(0xffffffffu, inc, o, 8);
                    if (tg >= o) inc += up;
                }
                const float pre = inc - tot;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    g[i][e] += pre;
                    if (fabsf(g[i][e]) > kLogDecayLimit) domain_ok = false;
                }
            }

            wait_phase_warp(sm.full[s], (n >> 1) & 1, abort);
            if (tg == 7)
#pragma unroll
                for (int e = 0; e < 8; ++e) S.gam[c0 + e] = expf(g[7][e]);
            if (pt < C) S.bet[pt] = bet;

            // a2: scaled operands, written over the landed tiles (same swizzle)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = 8 * tg + i;
                const uint32_t off = slab * 16384 + sw128_offset(t, col);
                const uint32_t offv = slab * 8192 + sw128_offset(t, col);
                float kf[8], qf[8], kh[8], qh[8], kb[8];
                if (t < valid) {
                    unpack8(*reinterpret_cast<const uint4 *>(S.kq + off), kf);
                    unpack8(*reinterpret_cast<const uint4 *>(S.kq + off + 8192), qf);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) kf[e] = qf[e] = 0.f;
                    *reinterpret_cast<uint4 *>(S.v + offv) = make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float gf = __expf(g[i][e]);
                    const float gi = __expf(-g[i][e]);
                    kh[e] = kf[e] * gf;
                    qh[e] = qf[e] * gf;
                    kb[e] = kf[e] * gi;
                }
                *reinterpret_cast<uint4 *>(S.kq + off) = pack8(kh);
                *reinterpret_cast<uint4 *>(S.kq + off + 8192) = pack8(qh);
                *reinterpret_cast<uint4 *>(S.kb + offv) = pack8(kb);
            }
            fence_proxy_async_smem();
            named_bar_sync(kBarPrep, 128);

            // a3 + a5: R = [Kh; Qh] Kb^T (M = 128, N = 64, K = 128)
            if (pt == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t a =
                        desc_sw128(smem_u32(S.kq) + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
                    const uint64_t b =
                        desc_sw128(smem_u32(S.kb) + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024);
                    mma_bf16(tmem + kColRW, a, b, id, k > 0);
                }
                mma_commit(smem_u32(&sm.bar_r));
            }
            wait_phase_warp(sm.bar_r, n & 1, abort);
            tc_fence_after();
            if (L < 64) {  // A[r][j] = beta_r R[r][j], j < r
                const int r = L;
                const float br = S.bet[r];
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t x[16];
                    tmem_ld16(tmem + lane_addr + kColRW + 16 * cb, x);
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        float4 w;
                        const int j = 16 * cb + 4 * j4;
                        w.x = j + 0 < r ? br * __uint_as_float(x[4 * j4 + 0]) : 0.f;
                        w.y = j + 1 < r ? br * __uint_as_float(x[4 * j4 + 1]) : 0.f;
                        w.z = j + 2 < r ? br * __uint_as_float(x[4 * j4 + 2]) : 0.f;
                        w.w = j + 3 < r ? br * __uint_as_float(x[4 * j4 + 3]) : 0.f;
                        *reinterpret_cast<float4 *>(&sm.as[r * LDA + j]) = w;
                    }
                }
            } else {  // M[r][j] = R[64 + r][j], j <= r
                const int r = L - 64;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t x[16];
                    tmem_ld16(tmem + lane_addr + kColRW + 16 * cb, x);
                    float f[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        f[j] = 16 * cb + j <= r ? __uint_as_float(x[j]) : 0.f;
                    store_row16(S.m, r, 16 * cb, f);
                }
            }
            tc_fence_before();
            named_bar_sync(kBarPrep, 128);

            // a4: T' = (I + A)^-1 diag(beta)
            solve_ut(sm, S.bet, pt);
            fence_proxy_async_smem();
            named_bar_sync(kBarPrep, 128);

            // a4: W^T = Kh^T T'^T, U~^T = V^T T'^T (M = 128, N = 64, K = 64)
            if (pt == 0) {
                if (n >= 2) wait_phase(sm.uempty[s], ((n >> 1) - 1) & 1, abort);
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, true, false);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t aw = desc_sw128(smem_u32(S.kq) + k * 2048, 16384, 1024);
                    const uint64_t av = desc_sw128(smem_u32(S.v) + k * 2048, 8192, 1024);
                    const uint64_t b = desc_sw128(smem_u32(sm.tp) + k * 32, 16, 1024);
                    mma_bf16(tmem + kColRW, aw, b, id, k > 0);
                    mma_bf16(tmem + kColU + 64 * s, av, b, id, k > 0);
                }
                mma_commit(smem_u32(&sm.bar_w));
            }
            wait_phase_warp(sm.bar_w, n & 1, abort);
            tc_fence_after();
            {  // -W as the MN-major operand [c][r], over the Kh area
                const int c = L;
                uint8_t *dst = S.kq + (c >> 6) * 16384;
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t x[16];
                    tmem_ld16(tmem + lane_addr + kColRW + 16 * cb, x);
                    float f[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) f[j] = -__uint_as_float(x[j]);
                    store_row16(dst, c & 63, 16 * cb, f);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(kBarPrep, 128);
            if (pt == 0) mbar_arrive(smem_u32(&sm.ready[s]));
        }
        if (!domain_ok) sm.domain = 1;
    } else {
        // -------------------------------------------------- serial carry (a6)
        const int et = tid - 32 * kEpiWarp0;
        const bool issuer = et == 0;
        const int v = L;
        {  // initial state: row v of S0 ([v][c] memory) -> TMEM fp32 and bf16 operand
            const float *src = p.S0 ? p.S0 + state_off + (size_t)v * D : nullptr;
#pragma unroll
            for (int cb = 0; cb < 8; ++cb) {
                float f[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float4 x = src ? reinterpret_cast<const float4 *>(src + 16 * cb)[q]
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    f[4 * q] = x.x; f[4 * q + 1] = x.y; f[4 * q + 2] = x.z; f[4 * q + 3] = x.w;
                }
                uint32_t u[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) u[j] = __float_as_uint(f[j]);
                tmem_st16(tmem + lane_addr + kColS + 16 * cb, u);
                store_row16(sm.sb + (cb >> 2) * 16384, v, 16 * (cb & 3), f);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(kBarEpi, 128);
        }

        auto issue_carry_in = [&](int n) {  // U^T += S^T (-W)^T ; O^T = S^T Qh^T
            const int s = n & 1;
            TcStage &S = sm.st[s];
            wait_phase(sm.ready[s], (n >> 1) & 1, abort);
            tc_fence_after();
            const uint32_t id_u = idesc_bf16(128, 64, false, true);
            const uint32_t id_o = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t a =
                    desc_sw128(smem_u32(sm.sb) + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
                const uint64_t bw =
                    desc_sw128(smem_u32(S.kq) + (k >> 2) * 16384 + (k & 3) * 2048, 8192, 1024);
                const uint64_t bq = desc_sw128(
                    smem_u32(S.kq) + 8192 + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
                mma_bf16(tmem + kColU + 64 * s, a, bw, id_u, 1);
                mma_bf16(tmem + kColO + 64 * s, a, bq, id_o, k > 0);
            }
            mma_commit(smem_u32(&sm.bar_u));
        };

        auto store_output = [&](int n) {  // O^T (lane v, column r) -> o[t0 + r][h][v]
            const int s = n & 1;
            const int64_t t0 = start + (int64_t)n * C;
            const int valid = min(C, len - n * C);
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t x[16];
                tmem_ld16(tmem + lane_addr + kColO + 64 * s + 16 * cb, x);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r = 16 * cb + j;
                    if (r < valid)
                        o[((size_t)(t0 + r) * p.H + h) * D + v] =
                            __float2bfloat16_rn(__uint_as_float(x[j]));
                }
            }
            tc_fence_before();
        };

        if (issuer) issue_carry_in(0);
        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            TcStage &S = sm.st[s];
            __syncwarp();  // the issuer lane rejoins before the warp-wide TMEM loads
            if (n >= 1) store_output(n - 1);
            wait_phase_warp(sm.bar_u, n & 1, abort);
            tc_fence_after();
            // U^T (lane v, column j) -> bf16 operand [v][j]
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t x[16];
                tmem_ld16(tmem + lane_addr + kColU + 64 * s + 16 * cb, x);
                float f[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(x[j]);
                store_row16(sm.ut, v, 16 * cb, f);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(kBarEpi, 128);
            if (issuer) {
                mbar_arrive(smem_u32(&sm.uempty[s]));
                tc_fence_after();
                const uint32_t id_o = idesc_bf16(128, 64, false, false);
                const uint32_t id_s = idesc_bf16(128, 128, false, true);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t a = desc_sw128(smem_u32(sm.ut) + k * 32, 16, 1024);
                    const uint64_t bm = desc_sw128(smem_u32(S.m) + k * 32, 16, 1024);
                    const uint64_t bk = desc_sw128(smem_u32(S.kb) + k * 2048, 8192, 1024);
                    mma_bf16(tmem + kColO + 64 * s, a, bm, id_o, 1);
                    mma_bf16(tmem + kColS, a, bk, id_s, 1);
                }
                mma_commit(smem_u32(&sm.bar_s));
                mma_commit(smem_u32(&sm.empty[s]));
            }
            wait_phase_warp(sm.bar_s, n & 1, abort);
            tc_fence_after();
            // S^T <- Diag(gamma) applied along c to (S^T + U^T Kb): TMEM fp32 and bf16 copy
#pragma unroll
            for (int cb = 0; cb < 8; ++cb) {
                uint32_t x[16];
                tmem_ld16(tmem + lane_addr + kColS + 16 * cb, x);
                float f[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    f[j] = __uint_as_float(x[j]) * S.gam[16 * cb + j];
                    x[j] = __float_as_uint(f[j]);
                }
                tmem_st16(tmem + lane_addr + kColS + 16 * cb, x);
                store_row16(sm.sb + (cb >> 2) * 16384, v, 16 * (cb & 3), f);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(kBarEpi, 128);
            if (issuer) {
                mbar_arrive(smem_u32(&sm.empty[s]));
                if (n + 1 < nchunks) issue_carry_in(n + 1);
            }
        }
        __syncwarp();
        store_output(nchunks - 1);
        if (p.S_T) {
            float *dst = p.S_T + state_off + (size_t)v * D;
#pragma unroll
            for (int cb = 0; cb < 8; ++cb) {
                uint32_t x[16];
                tmem_ld16(tmem + lane_addr + kColS + 16 * cb, x);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    reinterpret_cast<float4 *>(dst + 16 * cb)[q] =
                        make_float4(__uint_as_float(x[4 * q]), __uint_as_float(x[4 * q + 1]),
                                    __uint_as_float(x[4 * q + 2]), __uint_as_float(x[4 * q + 3]));
            }
        }
        tc_fence_before();
    }

    // ---------------------------------------------------------------- teardown
    if (tid == 32 * kPrepWarp0 || tid == 32 * kEpiWarp0) mma_commit(smem_u32(&sm.bar_fin));
    __syncthreads();
    if (tid == 0) {
        if (sm.abort) raise_status(p.status, KDA_ERR_TIMEOUT);
        else if (sm.domain) raise_status(p.status, KDA_ERR_DOMAIN);
    }
    if (warp == 0) {
        wait_drain(sm.bar_fin, 0);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// [Ttot][H][128] bf16 viewed as a 3-D tensor, tile = 64 channels x 1 head x 64 tokens.
bool make_token_map(CUtensorMap *map, const void *base, int H, int64_t Ttot) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)Ttot};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t elem[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(kda_dtype_t dt, int dk, int dv) {
    return dt == KDA_BF16 && dk == D && dv == D;
}

cudaError_t launch_prefill_tc(const FwdParams &p, cudaStream_t s) {
    if ((size_t)p.N * p.H == 0) return cudaSuccess;
    if (p.Ttot == 0) return launch_prefill_simt(p, KDA_BF16, s);  // nothing to contract
    if (p.Ttot > INT32_MAX) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv;
    if (!make_token_map(&mq, p.q, p.H, p.Ttot) || !make_token_map(&mk, p.k, p.H, p.Ttot) ||
        !make_token_map(&mv, p.v, p.H, p.Ttot))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(TcSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<<<(unsigned)((size_t)p.N * p.H), kThreads, smem, s>>>(p, mq, mk, mv);
    return cudaGetLastError();
}

}  // namespace kda

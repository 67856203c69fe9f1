// Tensor-core chunkwise KDA forward for sm_103a (bf16 q/k/v, d_k = d_v = 128).
//
// One CTA per (sequence, head) walks the sequence in 64-token chunks.  The
// algorithm is the chunk form of the recurrence (the CUDA-core engine gives the
// derivation; "Kimi Delta Attention 完全拆解", chunkwise section; "Kimi K3 的 KDA"
// section 5):
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
// tensor memory for the whole sequence (the S-update MMA accumulates into it),
// next to a bf16 copy that is the A operand of the carry-in MMAs, read straight
// from tensor memory.  The 64 x 64 triangular solve runs on the warp-level
// tensor cores (TF32, kda_solve.cuh).  Gates are handled in log2 units
// (G2 = G log2 e) so the exponentials are single ex2 instructions.
//
// Warp roles (384 threads, 3 warps per SM sub-partition, so up to 168
// registers per thread):
//   warps 0-7   chunk-local work of chunk n+1 (a1-a5): scaled operands, R and
//               its masks (all eight warps); the triangular solve (warps 0-3),
//               which writes T' in bf16 straight from its registers and so hands
//               the chunk to the carry warps, while warps 4-7 scan the gates of
//               the chunk after and park them in tensor memory.  Warp 0
//               allocates tensor memory; one thread loads each chunk's
//               log_alpha tile (TMA) as soon as the previous tile has been read.
//   warps 8-11  the serial carry of chunk n (a6): the W / U~ MMAs, -W out of
//               tensor memory into the operand tile, the U, O and S MMAs, the
//               gamma scaling of the state, and the output, staged in shared
//               memory and written with a TMA store.  One thread of the second
//               carry warp refills the q/k/v stage a chunk has just released
//               (TMA, 64 tokens x 64 channels per box, 128-byte swizzle) while
//               the MMA-issuing thread of the first sends the S update.
//               Issuing an MMA keeps a thread busy for about as long as the MMA
//               runs, so the W / U~ products are issued here, where the carry
//               would otherwise wait for the chunk-local warps.
// The chunk-local work of the next chunk overlaps the carry of the current one.
// kFullGrid (chosen by the launcher when nearly every SM holds a block) moves
// the bf16 stores of T''s diagonal blocks from the solve's first step to its
// idle warps in the second, which pays only on a busy GPU.
//
// kGated fuses the layer's output epilogue into the output stores: once the
// carry warps have staged a chunk's bf16 o tile, two threads per token read
// its row back, reduce its mean square over the 128 value channels (one
// shuffle joins the halves), read the gate logits from global memory and
// overwrite the row with y = sigmoid(g) w o / sqrt(mean(o^2) + eps) before
// the TMA store, so the unnormalised o never reaches HBM ("Kimi K3 模型结构（1）"
// output section: head-wise RMSNorm and sigmoid gate).
//
// Every mbarrier wait is bounded in time; on a timeout the kernel records
// KDA_ERR_TIMEOUT, runs its remaining steps without waiting, drains its own
// copies and MMAs, frees tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstddef>

#include "kda_internal.h"
#include "kda_sm100.cuh"
#include "kda_serial.cuh"
#include "kda_solve.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int D = 128;
constexpr int C = kChunk;
constexpr int kPrepWarp0 = 0, kPrepWarps = 8, kPrepThreads = 32 * kPrepWarps;
constexpr int kCarryWarp0 = 8, kCarryWarps = 4, kCarryThreads = 32 * kCarryWarps;
constexpr int kThreads = 32 * (kPrepWarps + kCarryWarps);
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns (fp32 accumulators, 128 lanes each)
constexpr uint32_t kColR = 0;     // R = [Kh; Qh] Kb^T        (64 columns)
constexpr uint32_t kColW = 64;    // W^T                      (64)
constexpr uint32_t kColU = 128;   // U~^T / U^T; later U^T in bf16 pairs (64)
constexpr uint32_t kColG = 192;   // G2 of the next chunk, parked between scan and scaling (64)
constexpr uint32_t kColO = 256;   // O^T                      (64)
constexpr uint32_t kColSb = 320;  // S^T, bf16 pairs          (64): MMA A operand
constexpr uint32_t kColS = 384;   // S^T master copy, fp32    (128)
constexpr int LDA = kSolveLd;     // fp32 row stride of the solve matrix
constexpr uint32_t kBarPrep = 1, kBarCarry = 2, kBarSolve = 3, kBarScan = 4;  // named barrier ids
constexpr uint32_t kTileBytes = 64 * 64 * 2;     // one TMA box
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLog2DecayLimit = kLogDecayLimit * kLog2e;

struct __align__(1024) TcStage {
    uint8_t kq[32768];  // per 64-channel slab: Kh rows 0-63 | Qh rows 0-63; Kh area -> -W
    uint8_t v[16384];   // V [token][v], two slabs
    uint8_t kb[16384];  // Kb [token][c], two slabs
    uint8_t m[8192];    // output mask [r][j]
    float gam[D];       // gamma per key channel
    float bet[C];       // beta per token (0 past the end)
    int wide;           // the chunk took the blocked path (kb holds K~, not Kb)
    uint8_t pad[252];
};

struct __align__(1024) TcSmem {
    TcStage st[2];
    uint8_t tp[8192];   // T' bf16 [r][j]; fp32 scratch while solving
    uint8_t ut[16384];  // the staged output tile [r][v] (two 64-channel slabs)
    uint8_t gt[32768];  // log_alpha tile: 4 boxes of 32 channels x 64 tokens (fp32, swizzled)
    float as[C * LDA];  // solve matrix / inverse blocks (fp32)
    uint64_t full[2], ready[2], gfull, tpfull;
    uint64_t bar_r, bar_u, bar_o, bar_s, bar_fin, tailfree[2];
    alignas(16) float wn[D];  // epilogue: the norm weight (ones when none is given), read as float4
    alignas(16) float bfac[6][D];  // blocked path: 2^(G2_16I - G2_16J) per key channel, J < I
    uint32_t tmem_base;
    int abort;
    int domain;
    int wide_chunk[2];  // scan -> chunk-local warps: chunk m (slot m % 2) takes the blocked path
};

// members read or written with 16-byte vector accesses
static_assert(sizeof(TcStage) == 74752, "stage layout");
static_assert(offsetof(TcSmem, wn) % 16 == 0 && offsetof(TcSmem, bfac) % 16 == 0 &&
                  offsetof(TcSmem, as) % 16 == 0 && offsetof(TcStage, gam) % 16 == 0 && offsetof(TcStage, bet) % 16 == 0,
              "16-byte vector accesses need 16-byte aligned members");

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

__device__ __forceinline__ uint4 pack8(const float *f) {
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                      pack_bf16(f[6], f[7]));
}

// Store n (multiple of 8) fp32 values as consecutive bf16 columns
// col .. col + n - 1 of one row of a 128-byte-swizzled tile.
template <int n>
__device__ __forceinline__ void store_row(uint8_t *tile, int row, int col, const float *f) {
#pragma unroll
    for (int j = 0; j < n; j += 8)
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, col + j)) = pack8(f + j);
}

// Gates of one prep thread from the landed log_alpha tile: tokens 2 l, 2 l + 1
// (l = lane) of channels c0 .. c0 + 15.  The tile is four TMA boxes of 32 fp32
// channels x 64 tokens with the 128-byte swizzle (16-byte chunk XOR row % 8).
__device__ __forceinline__ void read_gates(const uint8_t *gt, int lane, int fl, int c0,
                                           float (&g)[2][16]) {
    const uint8_t *box = gt + (c0 >> 5) * 8192;
    const int ch = (c0 & 31) >> 2;  // first of four 16-byte chunks in the 128-byte row
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int t = 2 * lane + (i ^ fl);
        const uint8_t *row = box + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(row + (((ch + k) ^ (t & 7)) << 4));
            g[i][4 * k + 0] = a.x;
            g[i][4 * k + 1] = a.y;
            g[i][4 * k + 2] = a.z;
            g[i][4 * k + 3] = a.w;
        }
    }
}

// T' = (I + A)^{-1} diag(beta) in bf16 ([r][j], 128-byte swizzle, into sm.tp)
// for the 64 x 64 strictly lower A in sm.as, on the warp-level tensor cores
// (kda_solve.cuh), written straight from the registers that produce it.
template <bool kOffloadDiag>
__device__ __forceinline__ void solve_ut(TcSmem &sm, const float *bet, int pt) {
    solve_tprime64<kOffloadDiag>(sm.as, bet, sm.tp, pt, kBarSolve);  // warps 0-3
}

// Pack 16 fp32 values (as bits) into 8 bf16 pairs (even index in the low half).
__device__ __forceinline__ void pack16(const uint32_t (&u)[16], uint32_t (&w)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = pack_bf16(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1]));
}

// d (16 x 8, fp32) += a (16 x 16) b (16 x 8), bf16 operands (warp-level tensor cores)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Token-serial pass over a whole (sequence, head), from S0: the fallback for a
// head with a chunk whose cumulative log-decay leaves [-80, 80] (kda_serial.cuh).
// Runs after teardown, over the block's shared memory: 64 tokens at a time are
// staged as fp32 by all 384 threads, threads 0-255 step through them with the
// state in registers, then all threads add the parts' output sums and store o.
// The chunk pass stored all its outputs (bulk wait, proxy fence) before the
// block barrier that precedes this, and they are overwritten here.
struct SerialStage {
    float k[C][D], q[C][D], a[C][D], v[C][D];
    float bet[C];
    float red_r[2 * Serial<D>::kParts * D];
    float red_o[C * Serial<D>::kParts * D];
};

template <bool kGated>
__device__ __forceinline__ void serial_head(const FwdParams *pp, uint8_t *smem_raw,
                                         int64_t start, int len, int h, const StateRef &sref) {
    const FwdParams &p = *pp;
    SerialStage &ss = *reinterpret_cast<SerialStage *>(
        smem_raw + ((16u - (smem_u32(smem_raw) & 15u)) & 15u));
    constexpr int CP = Serial<D>::kCP, P = Serial<D>::kParts;
    const int tid = threadIdx.x, vcol = tid % D, c0 = (tid / D) * CP;
    const bool stepper = tid < Serial<D>::kThreads;
    const bool vzero = sref.flags & kTaskVZero, no_out = sref.flags & kTaskNoOutput;
    const size_t n_tok = (size_t)p.Ttot * p.H * D, n_beta = (size_t)p.Ttot * p.H;
    const uint4 *q = static_cast<const uint4 *>(p.q);  // 8 bf16 per load; rows start on 16 bytes
    const uint4 *k = static_cast<const uint4 *>(p.k);
    const uint4 *v = static_cast<const uint4 *>(p.v);
    const float4 *la = reinterpret_cast<const float4 *>(p.log_alpha);
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
    // S[c0 + i][v] lives at memory [v][c0 + i]
    float st[CP];
    const size_t srow = sref.off + (size_t)vcol * D + c0;
#pragma unroll
    for (int i = 0; i < CP; ++i)
        st[i] = stepper && in_bounds(p.status, srow + i, sref.ext)
                    ? state_init(sref, vcol, c0 + i, D) : 0.f;
    for (int t0 = 0; t0 < len; t0 += C) {
        const int nt = min(C, len - t0);
        const size_t row0 = ((size_t)(start + t0) * p.H + h) * D;  // element index of token t0
        __syncthreads();  // the previous tokens' stage and output sums are read
        for (int idx = tid; idx < nt * (D / 8); idx += kThreads) {
            const int r = idx / (D / 8), c = (idx % (D / 8)) * 8;
            const size_t gi = row0 + (size_t)r * p.H * D + c;
            const bool ok = in_bounds(p.status, gi + 7, n_tok);
            float f[8];
            unpack8(ok ? k[gi / 8] : make_uint4(0, 0, 0, 0), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss.k[r][c + e] = f[e];
            unpack8(ok ? q[gi / 8] : make_uint4(0, 0, 0, 0), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss.q[r][c + e] = f[e];
            unpack8(ok && !vzero ? v[gi / 8] : make_uint4(0, 0, 0, 0), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss.v[r][c + e] = f[e];
        }
        for (int idx = tid; idx < nt * (D / 4); idx += kThreads) {
            const int r = idx / (D / 4), c = (idx % (D / 4)) * 4;
            const size_t gi = row0 + (size_t)r * p.H * D + c;
            const float4 g = in_bounds(p.status, gi + 3, n_tok) ? la[gi / 4]
                                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(&ss.a[r][c]) =
                make_float4(expf(g.x), expf(g.y), expf(g.z), expf(g.w));
        }
        if (tid < nt) {
            const size_t bi = (size_t)(start + t0 + tid) * p.H + h;
            ss.bet[tid] = in_bounds(p.status, bi, n_beta) ? p.beta[bi] : 0.f;
        }
        __syncthreads();
        if (stepper)
            serial_tokens<D, true, true>(st, &ss.k[0][0], &ss.q[0][0], &ss.a[0][0], &ss.v[0][0],
                                         ss.bet, D, nt, ss.red_r, ss.red_o, o, 0, 0, 0,
                                         p.status, 1);
        __syncthreads();
        if constexpr (kGated) {
            // one warp per token: the output epilogue over its 128 channels
            const int warp = tid >> 5, lane = tid & 31;
            const __nv_bfloat16 *gt = static_cast<const __nv_bfloat16 *>(p.gate);
            for (int r = warp; r < nt; r += kThreads / 32) {
                float ov[4], ssq = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int vv = lane + 32 * e;
                    ov[e] = 0.f;
#pragma unroll
                    for (int j = 0; j < P; ++j) ov[e] += ss.red_o[(r * P + j) * D + vv];
                    ssq = fmaf(ov[e], ov[e], ssq);
                }
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, m);
                const float rs = rsqrtf(ssq * (1.f / D) + p.eps);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int vv = lane + 32 * e;
                    const size_t oi = row0 + (size_t)r * p.H * D + vv;
                    if (in_bounds(p.status, oi, n_tok)) {
                        const float wv = p.norm_w ? p.norm_w[vv] : 1.f;
                        o[oi] = __float2bfloat16_rn(
                            ov[e] * rs * wv * sigmoid_bf16out(__bfloat162float(gt[oi])));
                    }
                }
            }
        } else {
            for (int idx = tid; idx < (no_out ? 0 : nt * D); idx += kThreads) {
                const int r = idx / D, vv = idx % D;
                float ov = 0.f;
#pragma unroll
                for (int j = 0; j < P; ++j) ov += ss.red_o[(r * P + j) * D + vv];
                const size_t oi = row0 + (size_t)r * p.H * D + vv;
                if (in_bounds(p.status, oi, n_tok)) o[oi] = __float2bfloat16_rn(ov);
            }
        }
    }
    if (stepper && sref.S_T) {
#pragma unroll
        for (int i = 0; i < CP; ++i)
            if (in_bounds(p.status, srow + i, sref.ext)) sref.S_T[srow + i] = st[i];
    }
}

// a3-a5 of a chunk on the blocked path (see the kernel): called by the 256
// threads of the chunk-local warps, which reach every named barrier inside.
// Out of line, so that the common path's code and registers do not change.
//
// For a chunk whose in-chunk log-decay leaves the chunk form's range (K3's
// per-token bound of -5 reaches -320 over 64 tokens), A and M are built in
// 16-token blocks, block I taking its decay reference at its first token 16 I
// (the scan checked that each block stays inside the range):
//   A[r][j] = beta_r sum_c Kh_rc Kb_jc,  M[r][j] = sum_c Qh_rc Kb_jc,  r in block I,
//   Kh = k 2^(G2_r - G2_16I) <= 1,  Qh likewise,  Kb = k 2^(G2_16I - G2_j),
// for j <= r ("Kimi K3 的 KDA" section 6 and "Kimi K3模型架构详解" section 3.4:
// with the decay bounded, sub-tiles with their own reference points keep every
// causal tile a dense product).  Kb of a token j of an earlier block J is its
// own block's Kb times 2^(G2_16I - G2_16J) <= 1, a per-channel factor, so one
// pass writes every operand once, each referenced to its own block: Kh and Qh
// over the landed k / q tile, Kb into the slot's kb area.  The 20 16 x 16 tiles
// of A and M (row block I, column block J <= I) then run at once on the
// warp-level tensor cores (bf16 m16n8k16, K = 128), the B fragments of a tile
// below the diagonal scaled by the factor table sm.bfac.  The fragment loads
// read the 128-byte-swizzled tiles conflict-free (eight rows, eight 16-byte
// columns).  Last, the chunk-start operands as on the other path, except K~ =
// k 2^(G2_63 - G2) <= 1 in place of Kb: the carry hands the state on as
// S <- Diag(gamma) S + K~^T U (scaling S before the product) instead of
// Diag(gamma) (S + Kb^T U), which would overflow here.  They are computed in
// the first pass and held in registers until the products have read the tiles.
template <bool kScaled>
__device__ __forceinline__ void blocked_tile(const TcSmem &sm, const TcStage &S, int mt, int I,
                                             int J, int lane, float (&acc)[2][4]) {
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint8_t *xa = S.kq + (mt ? 8192 : 0);
    const float *fac = sm.bfac[kScaled ? I * (I - 1) / 2 + J : 0];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int c = 16 * kk + 2 * t4, cc = c & 63;  // channel of a[0] / b0, its slab column
        const uint8_t *xs = xa + (kk >> 2) * 16384, *ys = S.kb + (kk >> 2) * 8192;
        uint32_t a[4];
        a[0] = *reinterpret_cast<const uint32_t *>(xs + sw128_offset(16 * I + g8, cc));
        a[1] = *reinterpret_cast<const uint32_t *>(xs + sw128_offset(16 * I + g8 + 8, cc));
        a[2] = *reinterpret_cast<const uint32_t *>(xs + sw128_offset(16 * I + g8, cc + 8));
        a[3] = *reinterpret_cast<const uint32_t *>(xs + sw128_offset(16 * I + g8 + 8, cc + 8));
        float2 f0, f1;
        if constexpr (kScaled) {
            f0 = *reinterpret_cast<const float2 *>(fac + c);
            f1 = *reinterpret_cast<const float2 *>(fac + c + 8);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int j = 16 * J + 8 * hh + g8;
            uint32_t b0 = *reinterpret_cast<const uint32_t *>(ys + sw128_offset(j, cc));
            uint32_t b1 = *reinterpret_cast<const uint32_t *>(ys + sw128_offset(j, cc + 8));
            if constexpr (kScaled) {
                b0 = pack_bf16(__uint_as_float(b0 << 16) * f0.x, __uint_as_float(b0 & 0xFFFF0000u) * f0.y);
                b1 = pack_bf16(__uint_as_float(b1 << 16) * f1.x, __uint_as_float(b1 & 0xFFFF0000u) * f1.y);
            }
            mma_bf16_16816(acc[hh], a, b0, b1);
        }
    }
}

// tiles of the products, (matrix << 4) | (I << 2) | J with matrix 0 = A, 1 = M:
// warp w takes entries w, w + 8 and w + 16: warps 0-3 the eight diagonal tiles
// (no factors) and one below the diagonal each, warps 4-7 two below it each
__constant__ uint8_t kBlockedTiles[20] = {
    0x00, 0x05, 0x0A, 0x0F, 0x04, 0x08, 0x09, 0x0C,  // A: (0,0) (1,1) (2,2) (3,3) | (1,0) (2,0) (2,1) (3,0)
    0x10, 0x15, 0x1A, 0x1F, 0x0D, 0x0E, 0x14, 0x18,  // M diagonal | A (3,1) (3,2), M (1,0) (2,0)
    0x19, 0x1C, 0x1D, 0x1E};                         // M (2,1) (3,0) (3,1) (3,2)

__device__ __noinline__ void blocked_chunk(TcSmem &sm, TcStage &S, uint32_t gaddr, int n,
                                           int valid, volatile int *abort) {
    const int pt = threadIdx.x, lane = pt & 31, pw = pt >> 5;
    const int s = n & 1;
    const int fl = (lane >> 2) & 1;
    const int c0 = 16 * pw;
    const int slab = c0 >> 6, col = c0 & 63;
    const int I = lane >> 3;  // the block of this thread's tokens 2 lane, 2 lane + 1
    // G2 of those tokens on channels c0 .. c0 + 15 is parked in tensor memory
    // (columns: slot 0's 16 channels, then slot 1's) and read as it is needed
    // no R product here: complete bar_r's phase of this chunk by hand, so that
    // the next chunk's wait on it keeps its parity
    if (pt == 0) {
        mbar_arrive(smem_u32(&sm.bar_r));
        S.wide = 1;  // for the carry, which clears it once it has read it
    }
    // G2 at the block's first token (lane 8 I, slot 0) and at token 63 (lane 31, slot 0)
    {  // factor table: lane 8 I + J (J < I) writes 2^(G2_16I - G2_16J) for this warp's channels
        const int J = lane & 7;
        uint32_t g0[16];
        tmem_ld16(gaddr, g0);
        float fi[16], fj[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            fi[e] = __shfl_sync(0xffffffffu, __uint_as_float(g0[e]), lane & 24);
            fj[e] = __shfl_sync(0xffffffffu, __uint_as_float(g0[e]), 8 * min(J, 3));
        }
        if (J < I) {
#pragma unroll
            for (int e = 0; e < 16; ++e) fj[e] = ex2_approx(fi[e] - fj[e]);
            float4 *dst = reinterpret_cast<float4 *>(sm.bfac[I * (I - 1) / 2 + J] + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = make_float4(fj[4 * q], fj[4 * q + 1], fj[4 * q + 2], fj[4 * q + 3]);
        }
    }
    // one pass over this thread's 2 tokens x 16 channels (8 channels at a
    // time): the block-referenced Kh, Qh (over the landed k / q tile) and Kb
    // (kb area), and the chunk-start Kh = k 2^G2, Qh and K~ as bf16 pairs,
    // parked in tensor memory until the products have read the tiles -- Kh and
    // Qh in this thread's 32 columns of the R accumulator (no R product on this
    // path), K~ over G2 columns 0-15 once each 8-column piece has been read;
    // column 8 k + 4 i (+ 16 for Qh) starts the pairs of slot i, channels c0 + 8 k ..
    const uint32_t park = gaddr - (kColG - kColR);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        uint32_t gk[2][8];  // G2 of slot i, channels c0 + 8 k ..
        tmem_ld8(gaddr + 8 * k, gk[0]);
        tmem_ld8(gaddr + 16 + 8 * k, gk[1]);
        // per channel: G2 at the block's first token (ref), 2^ref, and
        // 2^(G2_63 - ref + 64) for K~ = (Kb 2^-64) 2^(G2_63 - ref + 64): two
        // exact-range factors, since 2^(G2_63 - ref) alone can underflow while
        // K~ = k 2^(G2_63 - G2) is still a normal number
        float ref[8], pref[8], p63[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            ref[e] = __shfl_sync(0xffffffffu, __uint_as_float(gk[0][e]), lane & 24);
            const float g63 = __shfl_sync(0xffffffffu, __uint_as_float(gk[0][e]), 31);
            pref[e] = ex2_approx(ref[e]);
            p63[e] = ex2_approx(g63 - ref[e] + 64.f);
        }
        uint32_t khs[8], qhs[8], kts[8];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = 2 * lane + (i ^ fl);
            const uint32_t off = slab * 16384 + sw128_offset(t, col + 8 * k);
            const uint32_t offv = slab * 8192 + sw128_offset(t, col + 8 * k);
            float kf[8], qf[8], kh[8], qh[8], kb[8], ks[8], qs[8], kt[8];
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
                const float gr = __uint_as_float(gk[i][e]);
                const float up = ex2_approx(gr - ref[e]);
                kh[e] = kf[e] * up;
                qh[e] = qf[e] * up;
                kb[e] = kf[e] * ex2_approx(ref[e] - gr);
                kt[e] = kb[e] * 0x1p-64f * p63[e];
                // Gamma = 2^G2 (it underflows only where 2^ref does, below fp32's range)
                const float gam = up * pref[e];
                ks[e] = kf[e] * gam;
                qs[e] = qf[e] * gam;
                // gamma: token 63 closes the chunk, and lane 31 holds it in slot 0
                if (i == 0 && lane == 31) S.gam[c0 + 8 * k + e] = gam;
            }
            *reinterpret_cast<uint4 *>(S.kq + off) = pack8(kh);
            *reinterpret_cast<uint4 *>(S.kq + off + 8192) = pack8(qh);
            *reinterpret_cast<uint4 *>(S.kb + offv) = pack8(kb);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                khs[4 * i + e] = pack_bf16(ks[2 * e], ks[2 * e + 1]);
                qhs[4 * i + e] = pack_bf16(qs[2 * e], qs[2 * e + 1]);
                kts[4 * i + e] = pack_bf16(kt[2 * e], kt[2 * e + 1]);
            }
        }
        tmem_st8(park + 8 * k, khs);
        tmem_st8(park + 16 + 8 * k, qhs);
        tmem_st8(gaddr + 8 * k, kts);
    }
    // M is zero right of the block's columns: warp pw clears 16-byte piece pw
    // (columns 8 pw .. 8 pw + 7) of its rows from piece 2 (I + 1) on
    if (pw >= 2 * (I + 1)) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
            *reinterpret_cast<uint4 *>(S.m + sw128_offset(2 * lane + i, 8 * pw)) = make_uint4(0, 0, 0, 0);
    }
    tmem_wait_st();
    named_bar_sync(kBarPrep, kPrepThreads);  // operands, factors and beta are in place
    if (pt == 0) sm.wide_chunk[s] = 0;       // (every thread has read it)

    // the products: A (fp32, beta-scaled, where the solve reads it) and M
    // (bf16, diagonal included)
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll 1
    for (int u = pw; u < 20; u += kPrepWarps) {
        const int code = kBlockedTiles[u];
        const int mt = code >> 4, bi = (code >> 2) & 3, bj = code & 3;
        float acc[2][4] = {};
        if (bj < bi)
            blocked_tile<true>(sm, S, mt, bi, bj, lane, acc);
        else
            blocked_tile<false>(sm, S, mt, bi, bj, lane, acc);
        // rows r = 16 bi + g8 (acc 0, 1) and r + 8 (acc 2, 3); columns j, j + 1
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int j = 16 * bj + 8 * hh + 2 * t4;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = 16 * bi + g8 + 8 * rr;
                const float v0 = acc[hh][2 * rr], v1 = acc[hh][2 * rr + 1];
                if (mt == 0) {  // only j < r is ever read
                    const float br = S.bet[r];
                    *reinterpret_cast<float2 *>(&sm.as[r * LDA + j]) = make_float2(br * v0, br * v1);
                } else {
                    *reinterpret_cast<uint32_t *>(S.m + sw128_offset(r, j)) =
                        pack_bf16(j <= r ? v0 : 0.f, j + 1 <= r ? v1 : 0.f);
                }
            }
        }
    }
    named_bar_sync(kBarPrep, kPrepThreads);  // the block-referenced tiles are read

    // the chunk-start operands over them
    {
        uint32_t x[32], y[16];
        tmem_ld32(park, x);
        tmem_ld16(gaddr, y);
#pragma unroll
        for (int ik = 0; ik < 4; ++ik) {
            const int i = ik >> 1, k = ik & 1;
            const int t = 2 * lane + (i ^ fl);
            const uint32_t off = slab * 16384 + sw128_offset(t, col + 8 * k);
            const uint32_t offv = slab * 8192 + sw128_offset(t, col + 8 * k);
            const int q = 8 * k + 4 * i;
            *reinterpret_cast<uint4 *>(S.kq + off) = make_uint4(x[q], x[q + 1], x[q + 2], x[q + 3]);
            *reinterpret_cast<uint4 *>(S.kq + off + 8192) =
                make_uint4(x[16 + q], x[17 + q], x[18 + q], x[19 + q]);
            *reinterpret_cast<uint4 *>(S.kb + offv) = make_uint4(y[q], y[q + 1], y[q + 2], y[q + 3]);
        }
    }
    fence_proxy_async_smem();
    // the previous chunk's W and U~ products (issued by the carry warps) have
    // finished reading sm.tp, which the solve overwrites next
    if (pt == 0 && n >= 1) wait_phase(sm.ready[s ^ 1], ((n - 1) >> 1) & 1, abort);
    tc_fence_before();
    named_bar_sync(kBarPrep, kPrepThreads);
}

// kTasks: task-table mode (segment-parallel forward); the plain instantiation
// compiles none of its per-task choices.
template <bool kTasks, bool kFullGrid, bool kGated, bool kBlocked>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o,
                      const __grid_constant__ CUtensorMap tm_g,
                      const __grid_constant__ CUtensorMap tm_vz) {
    static_assert(!(kTasks && kGated), "the fused epilogue serves plain calls only");
    static_assert(!(kBlocked && (kTasks || kGated)), "the blocked path serves plain calls only");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Align by offsetting the shared-memory pointer itself (not through an
    // integer round trip), so the compiler keeps every access in the shared
    // address space.
    TcSmem &sm = *reinterpret_cast<TcSmem *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (*p.status == KDA_ERR_INVALID_ARGUMENT) return;  // set by the schedule kernel

    const int h = blockIdx.x % p.H;
    const int rank = blockIdx.x / p.H;
    const int nseq = p.order ? p.order[rank] : rank;
    int64_t start;
    int len;
    seq_range(p, nseq, start, len);
    const int nchunks = (len + C - 1) / C;
    StateRef sref;  // S0 / S_T block and task flags
    if constexpr (kTasks)
        sref = state_ref(p, nseq, h, D, D);
    else
        sref = {p.S0, p.S_T, ((size_t)nseq * p.H + h) * D * D, (size_t)p.N * p.H * D * D, 0};
    const bool no_out = kTasks && (sref.flags & kTaskNoOutput);
    // a task with v = 0 reads its V tiles through a map that only holds zeros
    const CUtensorMap *tmv = &tm_v;
    if constexpr (kTasks)
        if (sref.flags & kTaskVZero) tmv = &tm_vz;
    const size_t n_tok = (size_t)p.Ttot * p.H * D, n_beta = (size_t)p.Ttot * p.H;
    if (nchunks == 0) {  // empty sequence: the state passes through
        if (sref.S_T)
            for (int i = tid; i < D * D; i += kThreads)
                if (in_bounds(p.status, sref.off + i, sref.ext))
                    sref.S_T[sref.off + i] = state_init(sref, i / D, i % D, D);
        return;
    }

    volatile int *abort = &sm.abort;
    if (tid == 0) {
        sm.abort = 0;
        sm.domain = 0;
        sm.wide_chunk[0] = sm.wide_chunk[1] = 0;
        sm.st[0].wide = sm.st[1].wide = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.ready[s]), 1);
        }
        mbar_init(smem_u32(&sm.bar_r), 1);
        mbar_init(smem_u32(&sm.bar_u), 1);
        mbar_init(smem_u32(&sm.bar_s), 1);
        mbar_init(smem_u32(&sm.bar_o), 1);
        mbar_init(smem_u32(&sm.tailfree[0]), 1);
        mbar_init(smem_u32(&sm.tailfree[1]), 1);
        mbar_init(smem_u32(&sm.bar_fin), 2);
        mbar_init(smem_u32(&sm.gfull), 1);
        mbar_init(smem_u32(&sm.tpfull), 1);
        fence_mbar_init();
    }
    if constexpr (kGated)
        if (tid < D) sm.wn[tid] = p.norm_w ? p.norm_w[tid] : 1.f;
    if (warp == kPrepWarp0) {
        tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int L = 32 * (warp & 3) + lane;  // this thread's TMEM lane

    // TMA of the q, k, v tiles of chunk n into stage n % 2 (and an L2 prefetch of
    // the chunk after), and of the log_alpha tile of chunk n into the gate buffer.
    auto load_stage = [&](int n) {
        const int s = n & 1;
        const uint32_t fb = smem_u32(&sm.full[s]);
        mbar_arrive_expect_tx(fb, 6 * kTileBytes);
        const int t0 = static_cast<int>(start + (int64_t)n * C);
        TcStage &S = sm.st[s];
        tma_load_3d(smem_u32(S.kq), &tm_k, fb, 0, h, t0);
        tma_load_3d(smem_u32(S.kq + 8192), &tm_q, fb, 0, h, t0);
        tma_load_3d(smem_u32(S.kq + 16384), &tm_k, fb, 64, h, t0);
        tma_load_3d(smem_u32(S.kq + 24576), &tm_q, fb, 64, h, t0);
        tma_load_3d(smem_u32(S.v), tmv, fb, 0, h, t0);
        tma_load_3d(smem_u32(S.v + 8192), tmv, fb, 64, h, t0);
        if (n + 1 < nchunks) {
            const int t1 = t0 + C;
            tma_prefetch_3d(&tm_k, 0, h, t1);
            tma_prefetch_3d(&tm_k, 64, h, t1);
            tma_prefetch_3d(&tm_q, 0, h, t1);
            tma_prefetch_3d(&tm_q, 64, h, t1);
            if (tmv == &tm_v) {  // (the zero map holds nothing to prefetch)
                tma_prefetch_3d(&tm_v, 0, h, t1);
                tma_prefetch_3d(&tm_v, 64, h, t1);
            }
        }
    };
    auto load_gates = [&](int n) {
        const uint32_t gb = smem_u32(&sm.gfull);
        mbar_arrive_expect_tx(gb, 4 * 8192);
        const int t0 = static_cast<int>(start + (int64_t)n * C);
#pragma unroll
        for (int b = 0; b < 4; ++b) tma_load_3d(smem_u32(sm.gt + b * 8192), &tm_g, gb, 32 * b, h, t0);
    };
    if (tid == 32 * kCarryWarp0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_g);
        prefetch_tensormap(tmv);
        load_gates(0);
        load_stage(0);
        if (nchunks > 1) load_stage(1);
    }

    if (warp < kCarryWarp0) {
        // ------------------------------------------------ chunk-local work (a1-a5)
        const int pt = tid - 32 * kPrepWarp0;     // 0..255
        const int pw = pt >> 5;                   // prep warp 0..7
        const int half = pw >> 2;                 // which 32 of 64 TMEM columns
        // Scaled operands: warp pw owns channels 16 pw .. 16 pw + 15; lane l holds
        // tokens 2 l and 2 l + 1 of them.  Register slot i holds token
        // 2 l + (i ^ fl): lanes 4-7 of each group of 8 take the odd token first, so
        // the 8 lanes of a shared-memory phase touch 8 different rows mod 8 -- 8
        // different 16-byte columns of the swizzled tiles, free of bank conflicts.
        const int fl = (lane >> 2) & 1;
        const int c0 = 16 * pw;
        const int slab = c0 >> 6, col = c0 & 63;
        // Warps 4-7 scan the gates of the next chunk while warps 0-3 solve the
        // current one.  The scan uses the same layout (so the prefix sum over
        // tokens is one warp scan) for channel groups q and q + 4 (q = the warp's
        // TMEM quadrant, pw & 3) and parks G2 in tensor memory: quadrant q,
        // columns kColG (group q) and kColG + 32 (group q + 4).  Warp pw reads its
        // own group back from column kColG + 32 (pw >> 2).
        const bool scanner = pw >= 4;
        const int bt = pt - 128;
        const uint32_t gpark = tmem + lane_addr + kColG;

        // a1 for chunk m: log2-decay cumsum G2[t][c] = log2(e) sum_{t' <= t} log_alpha
        // of this thread's two tokens and the 16 channels from cg, from the landed
        // gate tile.
        auto gate_scan = [&](int m, int cg, float (&g)[2][16]) {
            const int validm = min(C, len - m * C);
            read_gates(sm.gt, lane, fl, cg, g);
            if (validm == C) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int e = 0; e < 16; e += 2) mul2(g[i][e], g[i][e + 1], kLog2e, kLog2e);
            } else {  // the tile runs past the sequence end
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const bool live = 2 * lane + (i ^ fl) < validm;
#pragma unroll
                    for (int e = 0; e < 16; ++e) g[i][e] = live ? g[i][e] * kLog2e : 0.f;
                }
            }
            // packed pairs of channels throughout (the same roundings as scalar
            // instructions, half the issue slots)
            float inc[16];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {  // this lane's total
                inc[e] = g[0][e];
                inc[e + 1] = g[0][e + 1];
                add2(inc[e], inc[e + 1], g[1][e], g[1][e + 1]);
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {  // inclusive scan across the warp
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const float up0 = __shfl_up_sync(0xffffffffu, inc[e], o);
                    const float up1 = __shfl_up_sync(0xffffffffu, inc[e + 1], o);
                    if (lane >= o) add2(inc[e], inc[e + 1], up0, up1);
                }
            }
            // slot i holds token 2 l + (i ^ fl): the odd token's G2 is the
            // inclusive sum, the even token's that minus the odd token's
            // log-decay -- as weights (one of fl, 1 - fl is 0) instead of
            // selects, with the same single rounding
            const float wf = fl ? 1.f : 0.f, wn = 1.f - wf;
            float amax = 0.f;  // largest |G2| of the odd tokens (the inclusive sums)
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                float s00 = inc[e], s01 = inc[e + 1], s10 = inc[e], s11 = inc[e + 1];
                fma2(s00, s01, -wn, -wn, g[1][e], g[1][e + 1]);  // slot 0
                fma2(s10, s11, -wf, -wf, g[0][e], g[0][e + 1]);  // slot 1
                g[0][e] = s00;
                g[0][e + 1] = s01;
                g[1][e] = s10;
                g[1][e + 1] = s11;
                amax = fmaxf(amax, fmaxf(fabsf(inc[e]), fabsf(inc[e + 1])));
            }
            // a chunk outside the chunk form's range takes the blocked path
            // (kBlocked: four 16-token blocks, each with its own decay
            // reference) when every block stays inside the range; otherwise
            // the whole (sequence, head) goes to the token-serial pass after
            // teardown.  G2 only decreases along the chunk, so a block's range
            // is G2 at its first token (lane 8 I, slot 0) minus G2 at its last
            // (lane 8 I + 7, slot 0).
            if constexpr (kBlocked) {
                if (__any_sync(0xffffffffu, !(amax <= kLog2DecayLimit))) {
                    float bmax = 0.f;
#pragma unroll
                    for (int I = 0; I < 4; ++I)
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float top = __shfl_sync(0xffffffffu, g[0][e], 8 * I);
                            const float bot = __shfl_sync(0xffffffffu, g[0][e], 8 * I + 7);
                            bmax = fmaxf(bmax, top - bot);
                        }
                    if (!(bmax <= kLog2DecayLimit))
                        *reinterpret_cast<volatile int *>(&sm.domain) = 1;
                    else
                        *reinterpret_cast<volatile int *>(&sm.wide_chunk[m & 1]) = 1;
                }
            } else if (!(amax <= kLog2DecayLimit)) {
                *reinterpret_cast<volatile int *>(&sm.domain) = 1;
            }
        };
        // Warps 4-7: gates of chunk m scanned and parked; once every scanning
        // thread has read the gate tile, it takes chunk m + 1.
        auto scan_ahead = [&](int m) {
            wait_phase_warp(sm.gfull, m & 1, abort);
#pragma unroll 1
            for (int h2 = 0; h2 < 2; ++h2) {  // channel groups q, then q + 4
                float gm[2][16];
                gate_scan(m, 16 * ((pw & 3) + 4 * h2), gm);
                tmem_st32(gpark + 32 * h2, reinterpret_cast<const uint32_t(&)[32]>(gm));
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(kBarScan, 128);
            if (bt == 96 && m + 1 < nchunks) load_gates(m + 1);
        };

        if (scanner) scan_ahead(0);
        float bn = 0.f;  // beta of the next chunk, loaded one chunk ahead
        if (pt < C && pt < len && in_bounds(p.status, (size_t)(start + pt) * p.H + h, n_beta))
            bn = p.beta[(size_t)(start + pt) * p.H + h];

        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            TcStage &S = sm.st[s];
            const int64_t t0 = start + (int64_t)n * C;
            const int valid = min(C, len - n * C);
            // G2 of chunk n, parked by warps 4-7 one step earlier
            named_bar_sync(kBarPrep, kPrepThreads);
            tc_fence_after();
            float g[2][16];
            tmem_ld32(gpark + 32 * half, reinterpret_cast<uint32_t(&)[32]>(g));
            const float bet = bn;
            if (n + 1 < nchunks) {
                const int valid1 = min(C, len - (n + 1) * C);
                const size_t bi = (size_t)(t0 + C + pt) * p.H + h;
                bn = (pt < C && pt < valid1 && in_bounds(p.status, bi, n_beta)) ? p.beta[bi] : 0.f;
            }

            // the scan of this chunk (one step earlier) chose the blocked path
            bool wide = false;
            if constexpr (kBlocked) wide = *reinterpret_cast<volatile int *>(&sm.wide_chunk[s]) != 0;

            wait_phase_warp(sm.full[s], (n >> 1) & 1, abort);
            // Kb, M and gamma of chunk n - 2 (same slot) are no longer read by the carry
            if (n >= 2) wait_phase_warp(sm.tailfree[s], ((n >> 1) - 1) & 1, abort);
            if (pt < C) S.bet[pt] = bet;

          if (!wide) {
            // a2: scaled operands, written over the landed tiles (same swizzle)
#pragma unroll
            for (int ik = 0; ik < 4; ++ik) {
                const int i = ik >> 1, k = ik & 1;
                const float *gr = g[i] + 8 * k;
                const int t = 2 * lane + (i ^ fl);
                const uint32_t off = slab * 16384 + sw128_offset(t, col + 8 * k);
                const uint32_t offv = slab * 8192 + sw128_offset(t, col + 8 * k);
                float kf[8], qf[8], kb[8], gfv[8];
                if (t < valid) {
                    unpack8(*reinterpret_cast<const uint4 *>(S.kq + off), kf);
                    unpack8(*reinterpret_cast<const uint4 *>(S.kq + off + 8192), qf);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) kf[e] = qf[e] = 0.f;
                    *reinterpret_cast<uint4 *>(S.v + offv) = make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float gf0 = ex2_approx(gr[e]), gf1 = ex2_approx(gr[e + 1]);
                    const float gi0 = ex2_approx(-gr[e]), gi1 = ex2_approx(-gr[e + 1]);
                    gfv[e] = gf0;
                    gfv[e + 1] = gf1;
                    kb[e] = kf[e];
                    kb[e + 1] = kf[e + 1];
                    mul2(kb[e], kb[e + 1], gi0, gi1);
                    mul2(kf[e], kf[e + 1], gf0, gf1);
                    mul2(qf[e], qf[e + 1], gf0, gf1);
                }
                *reinterpret_cast<uint4 *>(S.kq + off) = pack8(kf);
                *reinterpret_cast<uint4 *>(S.kq + off + 8192) = pack8(qf);
                *reinterpret_cast<uint4 *>(S.kb + offv) = pack8(kb);
                // gamma: token 63 closes the chunk, and lane 31 holds it in
                // slot 0 -- its Gamma, just computed, is the chunk's decay
                if (i == 0 && lane == 31) {
                    float4 *gd = reinterpret_cast<float4 *>(S.gam + c0 + 8 * k);
                    gd[0] = make_float4(gfv[0], gfv[1], gfv[2], gfv[3]);
                    gd[1] = make_float4(gfv[4], gfv[5], gfv[6], gfv[7]);
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(kBarPrep, kPrepThreads);

            // a3 + a5: R = [Kh; Qh] Kb^T (M = 128, N = 64, K = 128)
            if (pt == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, false, false);
                // one descriptor per operand; the k-th slice adds its byte offset
                // / 16 to the start-address field (no carry: shared addresses
                // stay far below 2^18)
                const uint64_t a0 = desc_sw128(smem_u32(S.kq), 16, 1024);
                const uint64_t b0 = desc_sw128(smem_u32(S.kb), 16, 1024);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16(tmem + kColR, a0 + (uint64_t)((k >> 2) * 1024 + (k & 3) * 2),
                             b0 + (uint64_t)((k >> 2) * 512 + (k & 3) * 2), id, k > 0);
                mma_commit(smem_u32(&sm.bar_r));
            }
            wait_phase_warp(sm.bar_r, n & 1, abort);
            tc_fence_after();
            {
                const int j0 = 32 * half;
                uint32_t x[32];
                tmem_ld32(tmem + lane_addr + kColR + j0, x);
                if (L < 64) {  // A[r][j] = beta_r R[r][j], j < r
                    const int r = L;
                    const float br = S.bet[r];
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const int j = j0 + 4 * j4;
                        float4 w = make_float4(__uint_as_float(x[4 * j4 + 0]), __uint_as_float(x[4 * j4 + 1]),
                                               __uint_as_float(x[4 * j4 + 2]), __uint_as_float(x[4 * j4 + 3]));
                        mul2(w.x, w.y, br, br);
                        mul2(w.z, w.w, br, br);
                        // stored in fp32 (the solve's tensor cores read the
                        // tf32 part); entries on and above the diagonal are
                        // never read by the solve, which overwrites them
                        *reinterpret_cast<float4 *>(&sm.as[r * LDA + j]) = w;
                    }
                } else {  // M[r][j] = R[64 + r][j], j <= r
                    const int r = L - 64;
                    float f[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        f[j] = j0 + j <= r ? __uint_as_float(x[j]) : 0.f;
                    store_row<32>(S.m, r, j0, f);
                }
            }
            // the previous chunk's W and U~ products (issued by the carry
            // warps) have finished reading sm.tp
            if (pt == 0 && n >= 1) wait_phase(sm.ready[s ^ 1], ((n - 1) >> 1) & 1, abort);
            tc_fence_before();
            named_bar_sync(kBarPrep, kPrepThreads);
          } else if constexpr (kBlocked) {
            blocked_chunk(sm, S, gpark + 32 * half, n, valid, abort);
          }

            if (!scanner) {
                // a4: T' = (I + A)^-1 diag(beta); the carry warps take it from here
                solve_ut<kFullGrid>(sm, S.bet, pt);
                fence_proxy_async_smem();
                named_bar_sync(kBarSolve, 128);
#if KDA_TEST_SKIP_ARRIVE
                // test-only build of the timeout path: chunk 1's T' is never
                // announced, so the carry's wait for it runs out of time
                if (pt == 0 && n != 1) mbar_arrive(smem_u32(&sm.tpfull));
#else
                if (pt == 0) mbar_arrive(smem_u32(&sm.tpfull));
#endif
            } else if (n + 1 < nchunks) {
                scan_ahead(n + 1);
            }
        }
    } else {
        // -------------------------------------------------- serial carry (a6)
        const int et = tid - 32 * kCarryWarp0;
        const bool issuer = et == 0;
        const int v = L;
        {  // initial state: row v of S0 ([v][c] memory) -> TMEM fp32 and bf16 operand
            const bool ident = kTasks && (sref.flags & kTaskS0Identity);
            const float *src =
                !ident && sref.S0 && in_bounds(p.status, sref.off + (size_t)v * D + D - 1, sref.ext)
                    ? sref.S0 + sref.off + (size_t)v * D
                    : nullptr;
#pragma unroll
            for (int cb = 0; cb < 8; ++cb) {
                uint32_t u[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float4 x = src ? reinterpret_cast<const float4 *>(src + 16 * cb)[q]
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ident) {  // row v of I: a one in column v
                        const int c = 16 * cb + 4 * q;
                        x = make_float4(c == v ? 1.f : 0.f, c + 1 == v ? 1.f : 0.f,
                                        c + 2 == v ? 1.f : 0.f, c + 3 == v ? 1.f : 0.f);
                    }
                    u[4 * q] = __float_as_uint(x.x); u[4 * q + 1] = __float_as_uint(x.y);
                    u[4 * q + 2] = __float_as_uint(x.z); u[4 * q + 3] = __float_as_uint(x.w);
                }
                tmem_st16(tmem + lane_addr + kColS + 16 * cb, u);
                uint32_t w[8];
                pack16(u, w);
                tmem_st8(tmem + lane_addr + kColSb + 8 * cb, w);
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(kBarCarry, kCarryThreads);
        }

        // O^T of chunk n (lane v, column r) -> staged tile [r][v] in sm.ut (two
        // 64-channel slabs, 128-byte swizzle) -> global: one TMA store per slab
        // for a full chunk; a masked copy for the last, partial chunk.
        // stage_output: O^T of chunk n (lane v, column r) -> staged bf16 tile,
        // which frees the O accumulator; finish_output: the epilogue (kGated)
        // and the store.  store_output does both.
        auto stage_output = [&](int n) {
            uint8_t *stage = sm.ut + (v >> 6) * 8192;
            const int vc = v & 63;
            // this column's byte offset in a row r of the swizzled tile depends
            // on r only through r % 8: eight bases, then constant offsets
            uint8_t *base[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) base[k] = stage + sw128_offset(k, vc) - k * 128;
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t x[32];
                tmem_ld32(tmem + lane_addr + kColO + 32 * cb, x);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int r = 32 * cb + j;
                    *reinterpret_cast<__nv_bfloat16 *>(base[r & 7] + (r >> 3) * 1024 + (r & 7) * 128) =
                        __float2bfloat16_rn(__uint_as_float(x[j]));
                }
            }
        };
        auto finish_output = [&](int n) {
            const int64_t t0 = start + (int64_t)n * C;
            const int valid = min(C, len - n * C);
            if constexpr (kGated) {
                // output epilogue over the staged bf16 tile (the caller has
                // synchronised the carry warps after staging), one row per two
                // threads: thread et takes token r = et / 2, channels
                // 64 (et % 2) .. + 63 (one 128-byte row of slab et % 2)
                const int r = et >> 1, half = et & 1;
                uint8_t *row = sm.ut + half * 8192 + (r >> 3) * 1024 + (r & 7) * 128;
                const bool live = r < valid;
                uint4 gq[8];
                const uint4 *gsrc = reinterpret_cast<const uint4 *>(
                    static_cast<const __nv_bfloat16 *>(p.gate) +
                    ((size_t)(t0 + (live ? r : 0)) * p.H + h) * D + 64 * half);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    gq[j] = live && in_bounds(p.status, ((size_t)(t0 + r) * p.H + h) * D + 64 * half + 8 * j + 7, n_tok)
                                ? gsrc[j] : make_uint4(0, 0, 0, 0);
                uint4 oq[8];
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    oq[j] = *reinterpret_cast<const uint4 *>(row + ((j ^ (r & 7)) << 4));
                    float f[8];
                    unpack8(oq[j], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);  // the row's other half
                const float rs = rsqrtf(ss * (1.f / D) + p.eps);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float f[8], gf[8];
                    unpack8(oq[j], f);
                    unpack8(gq[j], gf);
                    const float4 w0 = *reinterpret_cast<const float4 *>(&sm.wn[64 * half + 8 * j]);
                    const float4 w1 = *reinterpret_cast<const float4 *>(&sm.wn[64 * half + 8 * j + 4]);
                    const float wj[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = f[e] * (rs * wj[e]) * sigmoid_bf16out(gf[e]);
                    *reinterpret_cast<uint4 *>(row + ((j ^ (r & 7)) << 4)) = pack8(f);
                }
            }
            // every thread's writes to the tile are done and visible to the
            // async proxy before one thread hands it to the TMA store
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar_sync(kBarCarry, kCarryThreads);
            if (no_out) {
                // final state only: the tile was read out (freeing O) but is not stored
            } else if (valid == C) {
                if (issuer) {
                    tma_store_3d(&tm_o, smem_u32(sm.ut), 0, h, static_cast<int>(t0));
                    tma_store_3d(&tm_o, smem_u32(sm.ut + 8192), 64, h, static_cast<int>(t0));
                    bulk_commit_group();
                }
            } else {
                __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
                for (int idx = et; idx < valid * 16; idx += kCarryThreads) {
                    const int r = idx >> 4, ch = idx & 15;  // 16 pieces of 8 channels per row
                    const uint4 val = *reinterpret_cast<const uint4 *>(
                        sm.ut + (ch >> 3) * 8192 + sw128_offset(r, (ch & 7) * 8));
                    const size_t oi = ((size_t)(t0 + r) * p.H + h) * D + 8 * ch;
                    if (in_bounds(p.status, oi + 7, n_tok))
                        *reinterpret_cast<uint4 *>(o + oi) = val;
                }
            }
        };
        auto store_output = [&](int n) {
            stage_output(n);
            if constexpr (kGated) named_bar_sync(kBarCarry, kCarryThreads);
            finish_output(n);
        };

        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            TcStage &S = sm.st[s];
            if constexpr (kGated) {
                // the gate rows of chunk n into L2 (one 128-byte line per
                // thread): its epilogue reads them one chunk from now
                const int r = et >> 1;
                if (r < min(C, len - n * C))
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(
                        static_cast<const __nv_bfloat16 *>(p.gate) +
                        ((size_t)(start + (int64_t)n * C + r) * p.H + h) * D + 64 * (et & 1)));
            }
            // a4: W^T = Kh^T T'^T, U~^T = V^T T'^T (M = 128, N = 64, K = 64) once
            // the chunk-local warps have T'
            if (issuer) {
                wait_phase(sm.tpfull, n & 1, abort);
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, true, false);
                // (per slice k: the byte offset / 16 added to the start-address field)
                const uint64_t aw0 = desc_sw128(smem_u32(S.kq), 16384, 1024);
                const uint64_t av0 = desc_sw128(smem_u32(S.v), 8192, 1024);
                const uint64_t b0 = desc_sw128(smem_u32(sm.tp), 16, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t b = b0 + (uint64_t)(2 * k);
                    mma_bf16(tmem + kColW, aw0 + (uint64_t)(128 * k), b, id, k > 0);
                    mma_bf16(tmem + kColU, av0 + (uint64_t)(128 * k), b, id, k > 0);
                }
                mma_commit(smem_u32(&sm.ready[s]));
            }
            // W^T and U~^T of chunk n are complete: -W as the MN-major operand
            // [c][r] over the Kh area (lane c holds row c of W^T)
            __syncwarp();
            wait_phase_warp(sm.ready[s], (n >> 1) & 1, abort);
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t x[32];
                tmem_ld32(tmem + lane_addr + kColW + 32 * cb, x);
                // packed to bf16 pairs, then negated by flipping both sign bits
                uint8_t *tile = S.kq + (v >> 6) * 16384;
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(x[j]), __uint_as_float(x[j + 1])) ^ 0x80008000u;
                    w.y = pack_bf16(__uint_as_float(x[j + 2]), __uint_as_float(x[j + 3])) ^ 0x80008000u;
                    w.z = pack_bf16(__uint_as_float(x[j + 4]), __uint_as_float(x[j + 5])) ^ 0x80008000u;
                    w.w = pack_bf16(__uint_as_float(x[j + 6]), __uint_as_float(x[j + 7])) ^ 0x80008000u;
                    *reinterpret_cast<uint4 *>(tile + sw128_offset(v & 63, 32 * cb + j)) = w;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(kBarCarry, kCarryThreads);
            if (issuer) {  // U^T += S^T (-W)^T, S^T read from tensor memory
                tc_fence_after();
                const uint32_t id_u = idesc_bf16(128, 64, false, true);
                const uint64_t bw0 = desc_sw128(smem_u32(S.kq), 8192, 1024);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_tmem_a(tmem + kColU, tmem + kColSb + 8 * k,
                                    bw0 + (uint64_t)((k >> 2) * 1024 + (k & 3) * 128), id_u, 1);
                mma_commit(smem_u32(&sm.bar_u));
            }
            __syncwarp();
            // a chunk of the blocked path hands the state on as Diag(gamma) S + K~^T U:
            // scale the fp32 state now (the U and O products read its bf16 copy;
            // the S update below then adds K~^T U and scales by nothing)
            bool wide = false;
            if constexpr (kBlocked) wide = S.wide;
            if (wide) {
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t x[32];
                    tmem_ld32(tmem + lane_addr + kColS + 32 * cb, x);
                    const float4 *gm = reinterpret_cast<const float4 *>(S.gam + 32 * cb);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 gq = gm[q];
                        float a0 = __uint_as_float(x[4 * q + 0]), a1 = __uint_as_float(x[4 * q + 1]);
                        float a2 = __uint_as_float(x[4 * q + 2]), a3 = __uint_as_float(x[4 * q + 3]);
                        mul2(a0, a1, gq.x, gq.y);
                        mul2(a2, a3, gq.z, gq.w);
                        x[4 * q + 0] = __float_as_uint(a0);
                        x[4 * q + 1] = __float_as_uint(a1);
                        x[4 * q + 2] = __float_as_uint(a2);
                        x[4 * q + 3] = __float_as_uint(a3);
                    }
                    tmem_st32(tmem + lane_addr + kColS + 32 * cb, x);
                }
            }
            auto issue_o = [&] {  // O^T = S^T Qh^T
                if (issuer) {
                    tc_fence_after();
                    const uint32_t id_o = idesc_bf16(128, 64, false, false);
                    const uint64_t bq0 = desc_sw128(smem_u32(S.kq) + 8192, 16, 1024);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_bf16_tmem_a(tmem + kColO, tmem + kColSb + 8 * k,
                                        bq0 + (uint64_t)((k >> 2) * 1024 + (k & 3) * 2), id_o,
                                        k > 0);
                    mma_commit(smem_u32(&sm.bar_o));
                }
                __syncwarp();
            };
            if constexpr (kGated) {
                // the staged tile frees the O accumulator; the epilogue and the
                // store of chunk n - 1 then run while the U and O products do
                if (n >= 1) {
                    stage_output(n - 1);
                    tc_fence_before();
                    named_bar_sync(kBarCarry, kCarryThreads);
                }
                issue_o();
                if (n >= 1) finish_output(n - 1);
            } else {
                if (n >= 1) store_output(n - 1);  // frees the O accumulator
                issue_o();
            }
            wait_phase_warp(sm.bar_u, n & 1, abort);
            if (issuer) bulk_wait_group_read0();  // the previous output tile has left sm.ut
            named_bar_sync(kBarCarry, kCarryThreads);
            // a blocked chunk's gamma has been applied (every thread has read it):
            // ones for the S update below (ordered by its barrier)
            if (wide) {
                S.gam[et] = 1.f;
                if (et == 0) S.wide = 0;
            }
            tc_fence_after();
            // U^T (lane v, column j) -> bf16 pairs in tensor memory, over U^T itself:
            // the A operand of the two products that follow
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t x[32];
                tmem_ld32(tmem + lane_addr + kColU + 32 * cb, x);
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    w[j] = pack_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
                tmem_st16(tmem + lane_addr + kColU + 16 * cb, w);
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(kBarCarry, kCarryThreads);
            if (issuer) {
                tc_fence_after();
                const uint32_t id_o = idesc_bf16(128, 64, false, false);
                const uint32_t id_s = idesc_bf16(128, 128, false, true);
                const uint64_t bm0 = desc_sw128(smem_u32(S.m), 16, 1024);
                const uint64_t bk0 = desc_sw128(smem_u32(S.kb), 8192, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t a = tmem + kColU + 8 * k;
                    mma_bf16_tmem_a(tmem + kColO, a, bm0 + (uint64_t)(2 * k), id_o, 1);
                    mma_bf16_tmem_a(tmem + kColS, a, bk0 + (uint64_t)(128 * k), id_s, 1);
                }
                mma_commit(smem_u32(&sm.bar_s));
            } else if (et == 32 && n + 2 < nchunks) {
                // the U and O products (the last readers of the q / k / v tiles of
                // this slot) are done: refill it with chunk n + 2 while the carry
                // finishes chunk n (from a second warp, so that the copies go
                // out while the products above are being issued)
                wait_phase(sm.bar_o, n & 1, abort);
                load_stage(n + 2);
            }
            __syncwarp();
            wait_phase_warp(sm.bar_s, n & 1, abort);
            tc_fence_after();
            // S^T <- (S^T + U^T Kb) scaled by gamma along c: TMEM fp32 and bf16 copy
            // (for a blocked chunk gamma holds ones by now: its state is scaled)
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t x[32];
                tmem_ld32(tmem + lane_addr + kColS + 32 * cb, x);
                const float4 *gm = reinterpret_cast<const float4 *>(S.gam + 32 * cb);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 gq = gm[q];
                    float a0 = __uint_as_float(x[4 * q + 0]), a1 = __uint_as_float(x[4 * q + 1]);
                    float a2 = __uint_as_float(x[4 * q + 2]), a3 = __uint_as_float(x[4 * q + 3]);
                    mul2(a0, a1, gq.x, gq.y);
                    mul2(a2, a3, gq.z, gq.w);
                    x[4 * q + 0] = __float_as_uint(a0);
                    x[4 * q + 1] = __float_as_uint(a1);
                    x[4 * q + 2] = __float_as_uint(a2);
                    x[4 * q + 3] = __float_as_uint(a3);
                }
                tmem_st32(tmem + lane_addr + kColS + 32 * cb, x);
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    w[j] = pack_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
                tmem_st16(tmem + lane_addr + kColSb + 16 * cb, w);
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(kBarCarry, kCarryThreads);
            // Kb, M and gamma of this slot are no longer read: the chunk-local
            // warps may write chunk n + 2's
            if (issuer) mbar_arrive(smem_u32(&sm.tailfree[s]));
        }
        __syncwarp();
        store_output(nchunks - 1);
        if (issuer) {
            bulk_wait_group0();
            // order the bulk output stores before any later generic store to o
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        __syncwarp();
        // (every chunk's gates were scanned before its T' reached this warp, so
        // the flag is final here; a flagged head keeps S0 intact for the
        // token-serial pass, which writes S_T itself)
        if (sref.S_T && !*reinterpret_cast<volatile int *>(&sm.domain) &&
            in_bounds(p.status, sref.off + (size_t)v * D + D - 1, sref.ext)) {
            float *dst = sref.S_T + sref.off + (size_t)v * D;
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
    if (tid == 32 * kPrepWarp0 || tid == 32 * kCarryWarp0) mma_commit(smem_u32(&sm.bar_fin));
    if (tid == 32 * kCarryWarp0)  // never leave with a copy in flight
        for (int n = nchunks > 2 ? nchunks - 2 : 0; n < nchunks; ++n)
            wait_drain(sm.full[n & 1], (n >> 1) & 1);
    if (tid == 32 * kPrepWarp0) wait_drain(sm.gfull, (nchunks - 1) & 1);
    __syncthreads();
    if (tid == 0 && sm.abort) raise_status(p.status, KDA_ERR_TIMEOUT);
    if (warp == kPrepWarp0) {
        wait_drain(sm.bar_fin, 0);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (sm.domain && !sm.abort) serial_head<kGated>(&p, smem_raw, start, len, h, sref);
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

// SM count of the current device, looked up once per device (threads that
// race here all store the same value); 152 if the lookup fails.
int sm_count() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            return 152;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
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

// [Ttot][H][128] fp32 viewed as a 3-D tensor, tile = 32 channels x 1 head x 64
// tokens (128-byte rows, 128-byte swizzle).
bool make_gate_map(CUtensorMap *map, const float *base, int H, int64_t Ttot) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)Ttot};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
    cuuint32_t box[3] = {32, 1, 64};
    cuuint32_t elem[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides,
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
    CUtensorMap mq, mk, mv, mo, mg, mvz;
    if (!make_token_map(&mq, p.q, p.H, p.Ttot) || !make_token_map(&mk, p.k, p.H, p.Ttot) ||
        !make_token_map(&mv, p.v, p.H, p.Ttot) || !make_token_map(&mo, p.o, p.H, p.Ttot) ||
        !make_gate_map(&mg, p.log_alpha, p.H, p.Ttot))
        return cudaErrorInvalidValue;
    // V of kTaskVZero tasks: one head x 64 tokens of zeros; every other tile
    // coordinate lies outside it and is zero-filled by the copy
    if (p.vzero) {
        if (!make_token_map(&mvz, p.vzero, 1, 64)) return cudaErrorInvalidValue;
    } else {
        mvz = mv;
    }
    const size_t smem = sizeof(TcSmem) + 1024;
    // A grid that keeps (nearly) every SM busy runs the variant of the solve
    // whose bf16 diagonal blocks of T' are written by the idle warps of its
    // second step (5 % faster there, 1.5 % slower on fewer blocks; measured
    // on one head per SM for 96-304 blocks)
    const size_t blocks = (size_t)p.N * p.H;
    const bool full = blocks * 8 > (size_t)sm_count() * 7;
    if ((p.gate || p.blocked) && p.tasks) return cudaErrorInvalidValue;
    if (p.gate && p.blocked) return cudaErrorInvalidValue;
    auto kern = p.tasks     ? (full ? prefill_tc_kernel<true, true, false, false>
                                    : prefill_tc_kernel<true, false, false, false>)
                : p.gate    ? (full ? prefill_tc_kernel<false, true, true, false>
                                    : prefill_tc_kernel<false, false, true, false>)
                : p.blocked ? (full ? prefill_tc_kernel<false, true, false, true>
                                    : prefill_tc_kernel<false, false, false, true>)
                            : (full ? prefill_tc_kernel<false, true, false, false>
                                    : prefill_tc_kernel<false, false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, kThreads, smem, s>>>(p, mq, mk, mv, mo, mg, mvz);
    return cudaGetLastError();
}

}  // namespace kda

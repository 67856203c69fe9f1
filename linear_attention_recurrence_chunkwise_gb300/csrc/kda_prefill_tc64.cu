// Tensor-core chunkwise KDA forward for d_k = d_v = 64 (fp32 or bf16 q/k/v,
// fp32 state) on sm_103a, to fp32 accuracy.
//
// The chunk form of the 128-wide engine ("Kimi Delta Attention 完全拆解",
// chunkwise section; "Kimi K3 的 KDA" section 5), every contraction on tcgen05:
//
//   G = in-chunk inclusive cumsum of log_alpha, Gamma = exp(G), gamma = Gamma_63
//   Kh = K . Gamma,  Qh = Q . Gamma,  Kb = K / Gamma
//   R = [Kh; Qh] Kb^T:  A = StrictTril(diag(beta) R_top),  M = Tril(R_bottom)
//   [Z^T | O^T] = S^T [Kh; Qh]^T                    (issued with R, before the solve)
//   T' = (I + A)^-1 diag(beta)                      (fp32, by blocks)
//   U^T = (V^T - Z^T) T'^T,  O^T += U^T M^T,  S^T <- (S^T + U^T Kb) Diag(gamma)
//
// U = T' (V - Kh S) is the chunk form's U~ - W S with W = T' Kh and U~ = T' V,
// taken in the order that needs no W: the product with the state runs while
// the solve does, and one product follows it instead of two.
//
// fp32 accuracy from the bf16 tensor cores: each operand x is held as the pair
// hi = bf16(x), lo = bf16(x - hi), which leaves x - hi - lo within 2^-17 |x|,
// and each product is the sum of hi.hi, hi.lo and lo.hi over K slices of 16,
// accumulated in fp32 in tensor memory (the dropped lo.lo term is ~2^-16 of
// the product).  A pair takes the bytes of one fp32 operand: the hi and lo tiles
// of a 64-wide head have the shape of the two 64-channel slabs of a 128-wide
// bf16 head and use the same 128-byte-swizzled layouts and descriptors.
//
// Every MMA has M = 128: R stacks the Kh and Qh rows; the products whose left
// operand has 64 rows (S^T, V^T - Z^T and U^T, bf16 pairs read from tensor
// memory) hold them in lanes 64-127, so their results land in lanes 64-127, and
// lanes 0-63 of those operands stay zero.  So warps 0-1 (tensor-memory lanes
// 0-63) read out A, warps 2-3 (lanes 64-127) M, Z^T, U^T, O^T and the state.
//
// One CTA of 128 threads per (sequence, head) walks the chunks one at a time;
// one thread issues the MMAs and the TMA copies of the next chunk's rows (issued
// as soon as the current chunk's rows have been read, landing while the chunk
// computes).  The operand pass of the next chunk runs on warps 0-1 while warps
// 2-3 write out the current chunk's outputs and state: each thread takes two
// channels of 32 tokens (bf16 pairs packed two values per instruction, 32-bit
// stores).  The solve inverts the four 16 x 16 diagonal blocks of I + A by
// substitution, then assembles the two 32 x 32 halves and their lower-left
// block by fp32 block products over all four warps.
// A (sequence, head) with a chunk whose cumulative log-decay leaves [-80, 0]
// (exp(-G) past fp32 range) is recomputed token by token from S0 instead.
// Every mbarrier wait is bounded; a timeout records KDA_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int D = 64;
constexpr int C = kChunk;
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns (128 lanes each)
constexpr uint32_t kColR = 0;     // R = [Kh; Qh] Kb^T                    (64 fp32)
constexpr uint32_t kColZ = 64;    // Z^T, then U^T, in lanes 64-127       (64 fp32)
constexpr uint32_t kColO = 128;   // O^T in lanes 64-127                  (64 fp32)
static_assert(kColO == kColZ + 64, "[Z^T | O^T] is one product of N = 128");
constexpr uint32_t kColS = 192;   // S^T master in lanes 64-127           (64 fp32)
constexpr uint32_t kColSb = 256;  // S^T bf16 pairs: hi 32 columns, lo 32 (A operand)
constexpr uint32_t kColUb = 320;  // V^T - Z^T, then U^T, as bf16 pairs: hi 32 columns,
                                  // lo 32 (A operand)
constexpr int LDA = C + 4;        // fp32 row stride of A (rows start on 16 bytes)
constexpr int LDT = 36;           // fp32 row stride of the solve's 32 x 32 blocks

struct __align__(1024) Tc64Smem {
    uint8_t xq[32768];  // [Kh; Qh] K-major, 128 rows x 64 channels: hi tile | lo tile
    uint8_t kb[16384];  // Kb [j][c]: hi | lo; K-major B of R, MN-major B of the S update
    uint8_t tp[16384];  // T' [r][j] K-major: hi | lo
    uint8_t mm[16384];  // M [r][j] K-major: hi | lo
    float vt[C * D];    // V [t][v] in fp32 (for V^T - Z^T)
    float ts[4096];     // the solve's 32 x 32 blocks T1, T2 and P (fp32, rows of LDT)
    uint8_t raw[4 * C * 256];  // the next chunk's rows as they are in memory (TMA):
                               // log_alpha, k, q, v, 64 rows each of 64 elements
    float a[C * LDA];   // beta-scaled A (fp32); staging of the token-by-token pass
    float gpart[D];     // log2-decay sums of the first half of the chunk's tokens
    float gam[2][D];    // gamma of the chunk (even, odd)
    float bet[C];
    float rbet[C];      // the next chunk's beta (cp.async)
    uint64_t bar_mma, bar_fin, bar_ld, bar_zo;
    uint32_t tmem_base;
    int abort;
    int domain;
};

// Wait for a phase within the time limit, whatever the abort flag says (the
// teardown's waits for the last MMAs and the last row copy).
__device__ __forceinline__ void wait_bounded(uint64_t &bar, uint32_t parity) {
    if (mbar_try_wait(smem_u32(&bar), parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&bar), parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
}

// Global -> shared copy of 4 bytes that completes asynchronously (cp.async;
// waited for with cp_async_wait_all before a barrier).
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// byte offset of element (row, col) of a 64-column tile part (128-byte rows)
__device__ __forceinline__ uint32_t at(int row, int col) { return sw128_offset(row, col); }

// x0, x1 -> hi = their bf16 values as a pair (x0 in the low half) and lo =
// the bf16 pair of what is left (x - hi is exact in fp32), both rounded to
// nearest: one conversion instruction per pair
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

// columns col, col + 1 (col even) of one row of a tile pair whose lo part
// starts `part` bytes on
__device__ __forceinline__ void put2(uint8_t *tile, uint32_t part, int row, int col, float x0,
                                     float x1) {
    uint32_t h, l;
    split2(x0, x1, h, l);
    *reinterpret_cast<uint32_t *>(tile + at(row, col)) = h;
    *reinterpret_cast<uint32_t *>(tile + part + at(row, col)) = l;
}

// columns col .. col + 3 (col a multiple of 4) of one row of a tile pair
__device__ __forceinline__ void put4(uint8_t *tile, uint32_t part, int row, int col,
                                     const float4 &x) {
    uint32_t h0, l0, h1, l1;
    split2(x.x, x.y, h0, l0);
    split2(x.z, x.w, h1, l1);
    *reinterpret_cast<uint2 *>(tile + at(row, col)) = make_uint2(h0, h1);
    *reinterpret_cast<uint2 *>(tile + part + at(row, col)) = make_uint2(l0, l1);
}

// columns col .. col + 7 (col a multiple of 8) of one row of a tile pair
__device__ __forceinline__ void put8(uint8_t *tile, uint32_t part, int row, int col,
                                     const float *x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) split2(x[2 * i], x[2 * i + 1], h[i], l[i]);
    *reinterpret_cast<uint4 *>(tile + at(row, col)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(tile + part + at(row, col)) = make_uint4(l[0], l[1], l[2], l[3]);
}

// 32 fp32 values of a tensor-memory row -> 16 hi pairs and 16 lo pairs (the
// even K index in the low half), the A-operand format of the MMA
__device__ __forceinline__ void split_pairs(const uint32_t (&x)[32], uint32_t (&h)[16],
                                            uint32_t (&l)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        split2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]), h[i], l[i]);
}

// acc (4 columns) += x * the row y of a 32 x 32 block
__device__ __forceinline__ void axpy4(float4 &acc, float x, const float *y) {
    const float4 b = *reinterpret_cast<const float4 *>(y);
    acc.x = fmaf(x, b.x, acc.x);
    acc.y = fmaf(x, b.y, acc.y);
    acc.z = fmaf(x, b.z, acc.z);
    acc.w = fmaf(x, b.w, acc.w);
}

// The three-term product over K = 64: for each K slice g of 16, hi.hi, hi.lo,
// lo.hi.  Descriptors: base + part offset (hi 0, lo 1) + slice offset, in the
// 16-byte units of the start-address field.
__device__ __forceinline__ void mma3_ss(uint32_t d, uint64_t a0, uint32_t a_part, uint32_t a_k,
                                        uint64_t b0, uint32_t b_part, uint32_t b_k, uint32_t id,
                                        bool accumulate) {
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int term = 0; term < 3; ++term) {
            const uint32_t pa = term == 2, pb = term == 1;
            mma_bf16(d, a0 + (uint64_t)(pa * a_part + g * a_k), b0 + (uint64_t)(pb * b_part + g * b_k),
                     id, (accumulate || g || term) ? 1u : 0u);
        }
}

// The same with the left operand in tensor memory: pairs of part p, slice g at
// column a + 32 p + 8 g.
__device__ __forceinline__ void mma3_ts(uint32_t d, uint32_t a, uint64_t b0, uint32_t b_part,
                                        uint32_t b_k, uint32_t id, bool accumulate) {
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int term = 0; term < 3; ++term) {
            const uint32_t pa = term == 2, pb = term == 1;
            mma_bf16_tmem_a(d, a + 32 * pa + 8 * g, b0 + (uint64_t)(pb * b_part + g * b_k), id,
                            (accumulate || g || term) ? 1u : 0u);
        }
}

template <typename T>
__device__ __forceinline__ float ld(const T *p, size_t i) {
    if constexpr (sizeof(T) == 4)
        return p[i];
    else
        return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st(T *p, size_t i, float x) {
    if constexpr (sizeof(T) == 4)
        p[i] = x;
    else
        p[i] = __float2bfloat16_rn(x);
}

// Token-by-token pass over a whole (sequence, head) from its initial state, for
// a head with a chunk outside the chunk form's range: threads 0-63 each hold
// column v of S (S[c][v] for all c), the others stage the token.
template <typename T>
__device__ void serial_pass(const FwdParams &p, Tc64Smem &sm, int64_t start, int len, int h,
                            const StateRef &sref) {
    const int tid = threadIdx.x;
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    T *o = static_cast<T *>(p.o);
    const bool vzero = sref.flags & kTaskVZero, no_out = sref.flags & kTaskNoOutput;
    const size_t n_tok = (size_t)p.Ttot * p.H * D, n_beta = (size_t)p.Ttot * p.H;
    float *sk = sm.a, *sq = sm.a + D, *sa = sm.a + 2 * D, *sv = sm.a + 3 * D, *sb = sm.a + 4 * D;
    float s[D];
    const int vc = tid & (D - 1);
    const size_t srow = sref.off + (size_t)vc * D;
#pragma unroll
    for (int c = 0; c < D; ++c)
        s[c] = tid < D && in_bounds(p.status, srow + c, sref.ext) ? state_init(sref, vc, c, D) : 0.f;
    for (int t = 0; t < len; ++t) {
        const size_t row = ((size_t)(start + t) * p.H + h) * D;
        __syncthreads();  // the previous token's staging has been read
        if (tid < D) {
            const bool ok = in_bounds(p.status, row + tid, n_tok);
            sk[tid] = ok ? ld(k, row + tid) : 0.f;
            sq[tid] = ok ? ld(q, row + tid) : 0.f;
            sa[tid] = ok ? expf(p.log_alpha[row + tid]) : 1.f;
        } else {
            const int vv = tid - D;
            sv[vv] = !vzero && in_bounds(p.status, row + vv, n_tok) ? ld(v, row + vv) : 0.f;
            if (vv == 0) {
                const size_t bi = (size_t)(start + t) * p.H + h;
                sb[0] = in_bounds(p.status, bi, n_beta) ? p.beta[bi] : 0.f;
            }
        }
        __syncthreads();
        if (tid < D) {
            float r = 0.f;  // (alpha S)^T k
#pragma unroll
            for (int c = 0; c < D; ++c) {
                s[c] *= sa[c];
                r = fmaf(s[c], sk[c], r);
            }
            const float u = sb[0] * (sv[tid] - r);
            float ov = 0.f;
#pragma unroll
            for (int c = 0; c < D; ++c) {
                s[c] = fmaf(sk[c], u, s[c]);
                ov = fmaf(s[c], sq[c], ov);
            }
            if (!no_out && in_bounds(p.status, row + tid, n_tok)) st(o, row + tid, ov);
        }
    }
    if (tid < D && sref.S_T)
#pragma unroll
        for (int c = 0; c < D; ++c)
            if (in_bounds(p.status, srow + c, sref.ext)) sref.S_T[srow + c] = s[c];
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc64_kernel(const __grid_constant__ FwdParams p,
                        const __grid_constant__ CUtensorMap tm_la,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Tc64Smem &sm = *reinterpret_cast<Tc64Smem *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (*p.status == KDA_ERR_INVALID_ARGUMENT) return;  // set by the schedule kernel

    const int h = blockIdx.x % p.H;
    const int rank = blockIdx.x / p.H;
    const int nseq = p.order ? p.order[rank] : rank;
    int64_t start;
    int len;
    seq_range(p, nseq, start, len);
    const int nchunks = (len + C - 1) / C;
    const StateRef sref = state_ref(p, nseq, h, D, D);
    const bool vzero = sref.flags & kTaskVZero, no_out = sref.flags & kTaskNoOutput;
    const size_t n_tok = (size_t)p.Ttot * p.H * D, n_beta = (size_t)p.Ttot * p.H;
    if (nchunks == 0) {  // empty sequence: the state passes through
        if (sref.S_T)
            for (int i = tid; i < D * D; i += kThreads)
                if (in_bounds(p.status, sref.off + i, sref.ext))
                    sref.S_T[sref.off + i] = state_init(sref, i / D, i % D, D);
        return;
    }
    T *o = static_cast<T *>(p.o);

    volatile int *abort = &sm.abort;
    if (tid == 0) {
        sm.abort = 0;
        sm.domain = 0;
        mbar_init(smem_u32(&sm.bar_mma), 1);
        mbar_init(smem_u32(&sm.bar_fin), 1);
        mbar_init(smem_u32(&sm.bar_ld), 1);
        mbar_init(smem_u32(&sm.bar_zo), 1);
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
    const uint32_t lane_addr = static_cast<uint32_t>(32 * warp) << 16;
    const bool top = warp < 2;  // tensor-memory lanes 0-63
    const int L = 32 * warp + lane;
    uint32_t phase = 0;
    auto mma_done = [&] {  // every thread: the MMAs committed last have completed
        mbar_wait(smem_u32(&sm.bar_mma), phase & 1, abort);
        ++phase;
        tc_fence_after();
    };
    auto publish_smem = [&] {  // operand tiles written by threads -> the MMA issuer
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    };

    // initial state: lane 64 + v holds row v of S^T ([v][c] memory) in fp32 and
    // as bf16 pairs; lanes 0-63 of the pair columns are zero for good
    {
        uint32_t x[32], hp[16], lp[16];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (!top) {
                const int vv = L - 64;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const size_t i = sref.off + (size_t)vv * D + 32 * half + c;
                    x[c] = __float_as_uint(in_bounds(p.status, i, sref.ext)
                                               ? state_init(sref, vv, 32 * half + c, D) : 0.f);
                }
                split_pairs(x, hp, lp);
                tmem_st32(tmem + lane_addr + kColS + 32 * half, x);
            } else {
#pragma unroll
                for (int c = 0; c < 16; ++c) hp[c] = lp[c] = 0u;
                tmem_st16(tmem + lane_addr + kColUb + 16 * half, hp);
                tmem_st16(tmem + lane_addr + kColUb + 32 + 16 * half, lp);
            }
            tmem_st16(tmem + lane_addr + kColSb + 16 * half, hp);
            tmem_st16(tmem + lane_addr + kColSb + 32 + 16 * half, lp);
        }
        tmem_wait_st();
    }

    const uint32_t a_xq = smem_u32(sm.xq), a_kb = smem_u32(sm.kb);
    const uint32_t a_tp = smem_u32(sm.tp), a_mm = smem_u32(sm.mm);
    const uint32_t id_kk = idesc_bf16(128, 64, false, false);   // K-major A and B
    const uint32_t id_kk2 = idesc_bf16(128, 128, false, false); // the same, N = 128
    const uint32_t id_km = idesc_bf16(128, 64, false, true);    // MN-major B

    // chunk m's rows of log_alpha, k, q, v -> sm.raw by TMA (thread 0; tiles of
    // 64 tokens x one head x 64 channels, zero past the last token; rows past
    // the sequence's end belong to the next one and are masked when read) and
    // its beta -> sm.rbet (cp.async, threads t < rows of the chunk)
    const float *raw_la = reinterpret_cast<const float *>(sm.raw);
    const T *raw_k = reinterpret_cast<const T *>(sm.raw + C * 256);
    const T *raw_q = reinterpret_cast<const T *>(sm.raw + 2 * C * 256);
    const T *raw_v = reinterpret_cast<const T *>(sm.raw + 3 * C * 256);
    constexpr uint32_t kTile = C * D * sizeof(T);
    int ld_issued = 0;  // row copies issued by thread 0 (one bar_ld phase each)
    auto issue_rows = [&](int m) {
#if KDA_TEST_SKIP_ARRIVE
        if (m == 1) return;  // test-only build: chunk 1's rows never arrive, so its wait runs out
#endif
        const int tm = (int)(start + (int64_t)m * C);
        const uint32_t bar = smem_u32(&sm.bar_ld);
        mbar_arrive_expect_tx(bar, C * D * 4 + (vzero ? 2 : 3) * kTile);
        tma_load_3d(smem_u32(sm.raw), &tm_la, bar, 0, h, tm);
        tma_load_3d(smem_u32(sm.raw + C * 256), &tm_k, bar, 0, h, tm);
        tma_load_3d(smem_u32(sm.raw + 2 * C * 256), &tm_q, bar, 0, h, tm);
        if (!vzero) tma_load_3d(smem_u32(sm.raw + 3 * C * 256), &tm_v, bar, 0, h, tm);
        ++ld_issued;
    };
    auto stage_beta = [&](int m) {
        const int64_t tm = start + (int64_t)m * C;
        if (tid < min(C, len - m * C)) {
            const size_t bi = (size_t)(tm + tid) * p.H + h;
            if (in_bounds(p.status, bi, n_beta)) cp_async4(&sm.rbet[tid], p.beta + bi);
        }
    };
    if (tid == 0) {
        prefetch_tensormap(&tm_la);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_v);
        issue_rows(0);
    }
    // ------------------------------------------------ a1, a2: gates and operands
    // of chunk m, by warps 0-1 (the first chunk's before the loop, every other
    // one while warps 2-3 write out the chunk before it): thread (w, c2) takes
    // channels 2 c2, 2 c2 + 1 of tokens 32 w .. 32 w + 31 -- their log2-decays
    // summed per half first (the second half starts from the first half's
    // sum), then Gamma and 1 / Gamma by ex2 on the cumulative log2-decay, and
    // k, q as bf16 pairs, two channels per 32-bit store, v in fp32; thread t
    // takes the beta of token t.
    auto operands = [&](int m) {
        const int valid = min(C, len - m * C);
        const int c2 = tid & 31, w = tid >> 5, c = 2 * c2;
        constexpr float kLog2e = 1.4426950408889634f;
        mbar_wait(smem_u32(&sm.bar_ld), m & 1, abort);
        cp_async_wait_all();  // this thread's beta copy
        sm.bet[tid] = tid < valid ? sm.rbet[tid] : 0.f;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
            const int t = 32 * w + i;
            if (t < valid) {
                const float2 la = *reinterpret_cast<const float2 *>(raw_la + t * D + c);
                s0 = fmaf(la.x, kLog2e, s0);
                s1 = fmaf(la.y, kLog2e, s1);
            }
        }
        if (w == 0) *reinterpret_cast<float2 *>(&sm.gpart[c]) = make_float2(s0, s1);
        named_bar_sync(1, 64);
        float G0 = 0.f, G1 = 0.f;
        if (w) {
            const float2 g = *reinterpret_cast<const float2 *>(&sm.gpart[c]);
            G0 = g.x;
            G1 = g.y;
        }
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
            const int t = 32 * w + i;
            const bool live = t < valid;
            float k0 = 0.f, k1 = 0.f, q0 = 0.f, q1 = 0.f, v0 = 0.f, v1 = 0.f;
            if (live) {
                const float2 la = *reinterpret_cast<const float2 *>(raw_la + t * D + c);
                G0 = fmaf(la.x, kLog2e, G0);
                G1 = fmaf(la.y, kLog2e, G1);
                if constexpr (sizeof(T) == 4) {
                    const float2 kk = *reinterpret_cast<const float2 *>(raw_k + t * D + c);
                    const float2 qq = *reinterpret_cast<const float2 *>(raw_q + t * D + c);
                    k0 = kk.x, k1 = kk.y, q0 = qq.x, q1 = qq.y;
                    if (!vzero) {
                        const float2 vv = *reinterpret_cast<const float2 *>(raw_v + t * D + c);
                        v0 = vv.x, v1 = vv.y;
                    }
                } else {
                    const uint32_t kk = *reinterpret_cast<const uint32_t *>(raw_k + t * D + c);
                    const uint32_t qq = *reinterpret_cast<const uint32_t *>(raw_q + t * D + c);
                    k0 = __uint_as_float(kk << 16), k1 = __uint_as_float(kk & 0xFFFF0000u);
                    q0 = __uint_as_float(qq << 16), q1 = __uint_as_float(qq & 0xFFFF0000u);
                    if (!vzero) {
                        const uint32_t vv = *reinterpret_cast<const uint32_t *>(raw_v + t * D + c);
                        v0 = __uint_as_float(vv << 16), v1 = __uint_as_float(vv & 0xFFFF0000u);
                    }
                }
            }
            const float g0 = ex2_approx(G0), g1 = ex2_approx(G1);
            const float r0 = ex2_approx(-G0), r1 = ex2_approx(-G1);
            put2(sm.xq, 16384, t, c, k0 * g0, k1 * g1);
            put2(sm.xq, 16384, 64 + t, c, q0 * g0, q1 * g1);
            put2(sm.kb, 8192, t, c, k0 * r0, k1 * r1);
            *reinterpret_cast<float2 *>(&sm.vt[t * D + c]) = make_float2(v0, v1);
            if (t == C - 1) *reinterpret_cast<float2 *>(&sm.gam[m & 1][c]) = make_float2(g0, g1);
        }
        constexpr float kLimit2 = kLogDecayLimit * kLog2e;
        if (w == 1 && !(G0 >= -kLimit2 && G1 >= -kLimit2))
            *reinterpret_cast<volatile int *>(&sm.domain) = 1;
    };
    stage_beta(0);
    if (tid < 64) operands(0);
    publish_smem();

    for (int n = 0; n < nchunks; ++n) {
        const int64_t t0 = start + (int64_t)n * C;
        const int valid = min(C, len - n * C);
        if (*reinterpret_cast<volatile int *>(&sm.domain)) break;  // (read by all after the barrier)
        // the staged rows have been read: the next chunk's may land
        if (n + 1 < nchunks) {
            if (tid == 0 && !*abort) issue_rows(n + 1);
            stage_beta(n + 1);
        }

        // ---------------------------------------------- a3, a5: R = [Kh; Qh] Kb^T,
        // then [Z^T | O^T] = S^T [Kh; Qh]^T (completes on its own barrier)
        if (tid == 0) {
            tc_fence_after();
            mma3_ss(tmem + kColR, desc_sw128(a_xq, 16, 1024), 1024, 2, desc_sw128(a_kb, 16, 1024),
                    512, 2, id_kk, false);
            mma_commit(smem_u32(&sm.bar_mma));
            mma3_ts(tmem + kColZ, tmem + kColSb, desc_sw128(a_xq, 16, 1024), 1024, 2, id_kk2,
                    false);
            mma_commit(smem_u32(&sm.bar_zo));
        }
        __syncwarp();
        mma_done();
        {
            uint32_t x[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(tmem + lane_addr + kColR + 32 * half, x);
                if (top) {  // A[r][j] = beta_r R[r][j]; only j < r is read
                    const float br = sm.bet[L];
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(&sm.a[L * LDA + 32 * half + j]) =
                            make_float4(br * __uint_as_float(x[j]), br * __uint_as_float(x[j + 1]),
                                        br * __uint_as_float(x[j + 2]),
                                        br * __uint_as_float(x[j + 3]));
                } else {    // M[r][j] = R[64 + r][j], j <= r
                    const int r = L - 64;
#pragma unroll
                    for (int j8 = 0; j8 < 32; j8 += 8) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = 32 * half + j8 + e;
                            f[e] = j <= r ? __uint_as_float(x[j8 + e]) : 0.f;
                        }
                        put8(sm.mm, 8192, r, 32 * half + j8, f);
                    }
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---------------------------------------------- a4: T' = (I + A)^-1 diag(beta)
        // T = (I + A)^-1 by blocks: the four 16 x 16 diagonal blocks D_b by
        // forward substitution; the two 32 x 32 diagonal halves T1 = [D0 0; E0 D1]
        // and T2 = [D2 0; E1 D3] with E0 = -D1 (A10 D0), E1 = -D3 (A32 D2); the
        // lower-left half T21 = -T2 (A21 T1), in fp32.  Meanwhile warps 2-3 form
        // V^T - Z^T as bf16 pairs, the left operand of U^T.
        {
            float *T1 = sm.ts, *T2 = T1 + 32 * LDT, *P = T2 + 32 * LDT;
            if (tid < 64) {  // column jj of D_b: y = (I + A_bb)^-1 e_jj
                const int b = tid >> 4, jj = tid & 15;
                const float *Ab = sm.a + 16 * b * LDA + 16 * b;
                float y[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float acc = i == jj ? 1.f : 0.f;
#pragma unroll
                    for (int s4 = 0; s4 < i; s4 += 4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(Ab + i * LDA + s4);
                        acc = fmaf(-a4.x, y[s4], acc);
                        if (s4 + 1 < i) acc = fmaf(-a4.y, y[s4 + 1], acc);
                        if (s4 + 2 < i) acc = fmaf(-a4.z, y[s4 + 2], acc);
                        if (s4 + 3 < i) acc = fmaf(-a4.w, y[s4 + 3], acc);
                    }
                    y[i] = acc;
                }
                float *Db = (b < 2 ? T1 : T2) + (b & 1) * 16 * (LDT + 1);
#pragma unroll
                for (int i = 0; i < 16; ++i) Db[i * LDT + jj] = y[i];
            } else {  // V^T - Z^T (lane 64 + v: row v), and the zero upper-right
                      // blocks of T1 and T2
                mbar_wait(smem_u32(&sm.bar_zo), n & 1, abort);
                tc_fence_after();
                const int vv = L - 64;
                uint32_t x[32], hp[16], lp[16];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(tmem + lane_addr + kColZ + 32 * half, x);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        x[j] = __float_as_uint(sm.vt[(32 * half + j) * D + vv] - __uint_as_float(x[j]));
                    split_pairs(x, hp, lp);
                    tmem_st16(tmem + lane_addr + kColUb + 16 * half, hp);
                    tmem_st16(tmem + lane_addr + kColUb + 32 + 16 * half, lp);
                }
                tmem_wait_st();
                const int u = tid - 64;
#pragma unroll
                for (int e = u; e < 128; e += 64)
                    *reinterpret_cast<float4 *>((e < 64 ? T1 : T2) + ((e >> 2) & 15) * LDT + 16 +
                                                4 * (e & 3)) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncthreads();
            // thread (m, rr, cq): row rr, columns 4 cq .. 4 cq + 3 of the 16 x 16
            // product m (0: the T1 half, 1: the T2 half)
            const int m = tid >> 6, rr = (tid >> 2) & 15, cq = tid & 3;
            float *Tm = m ? T2 : T1;
            {  // P_m = A_(2m+1, 2m) D_2m  -> rows 16 m .. of P
                const float *x = sm.a + (16 + 32 * m + rr) * LDA + 32 * m;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k4 = 0; k4 < 16; k4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(x + k4);
                    axpy4(acc, a4.x, Tm + (k4 + 0) * LDT + 4 * cq);
                    axpy4(acc, a4.y, Tm + (k4 + 1) * LDT + 4 * cq);
                    axpy4(acc, a4.z, Tm + (k4 + 2) * LDT + 4 * cq);
                    axpy4(acc, a4.w, Tm + (k4 + 3) * LDT + 4 * cq);
                }
                *reinterpret_cast<float4 *>(P + (16 * m + rr) * LDT + 4 * cq) = acc;
            }
            __syncthreads();
            {  // E_m = -D_(2m+1) P_m  -> rows 16 .. 31, columns 0 .. 15 of the half
                const float *x = Tm + (16 + rr) * LDT + 16;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k4 = 0; k4 < 16; k4 += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(x + k4);
                    axpy4(acc, d4.x, P + (16 * m + k4 + 0) * LDT + 4 * cq);
                    axpy4(acc, d4.y, P + (16 * m + k4 + 1) * LDT + 4 * cq);
                    axpy4(acc, d4.z, P + (16 * m + k4 + 2) * LDT + 4 * cq);
                    axpy4(acc, d4.w, P + (16 * m + k4 + 3) * LDT + 4 * cq);
                }
                *reinterpret_cast<float4 *>(Tm + (16 + rr) * LDT + 4 * cq) =
                    make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
            }
            __syncthreads();
            // thread (rp, cq8): rows 2 rp, 2 rp + 1, columns 4 cq8 .. 4 cq8 + 3 of a
            // 32 x 32 block
            const int rp = tid >> 3, cq8 = tid & 7;
            const int r0 = 2 * rp, col = 4 * cq8;
            {  // P = A21 T1
                const float *x0 = sm.a + (32 + r0) * LDA, *x1 = x0 + LDA;
                float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll
                for (int k4 = 0; k4 < 32; k4 += 4) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(x0 + k4);
                    const float4 a1 = *reinterpret_cast<const float4 *>(x1 + k4);
                    const float *y = T1 + k4 * LDT + col;
                    axpy4(acc0, a0.x, y);
                    axpy4(acc1, a1.x, y);
                    axpy4(acc0, a0.y, y + LDT);
                    axpy4(acc1, a1.y, y + LDT);
                    axpy4(acc0, a0.z, y + 2 * LDT);
                    axpy4(acc1, a1.z, y + 2 * LDT);
                    axpy4(acc0, a0.w, y + 3 * LDT);
                    axpy4(acc1, a1.w, y + 3 * LDT);
                }
                *reinterpret_cast<float4 *>(P + r0 * LDT + col) = acc0;
                *reinterpret_cast<float4 *>(P + (r0 + 1) * LDT + col) = acc1;
            }
            __syncthreads();
            {  // T21 = -T2 P, and T' = T diag(beta) written as bf16 pairs: rows
               // 0-31 [T1 0], rows 32-63 [T21 T2]
                const float *x0 = T2 + r0 * LDT, *x1 = x0 + LDT;
                float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll
                for (int k4 = 0; k4 < 32; k4 += 4) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(x0 + k4);
                    const float4 a1 = *reinterpret_cast<const float4 *>(x1 + k4);
                    const float *y = P + k4 * LDT + col;
                    axpy4(acc0, a0.x, y);
                    axpy4(acc1, a1.x, y);
                    axpy4(acc0, a0.y, y + LDT);
                    axpy4(acc1, a1.y, y + LDT);
                    axpy4(acc0, a0.z, y + 2 * LDT);
                    axpy4(acc1, a1.z, y + 2 * LDT);
                    axpy4(acc0, a0.w, y + 3 * LDT);
                    axpy4(acc1, a1.w, y + 3 * LDT);
                }
                const float4 bl = *reinterpret_cast<const float4 *>(&sm.bet[col]);
                const float4 bh = *reinterpret_cast<const float4 *>(&sm.bet[32 + col]);
                auto scaled = [](const float4 &t, const float4 &b, float sg) {
                    return make_float4(sg * t.x * b.x, sg * t.y * b.y, sg * t.z * b.z, sg * t.w * b.w);
                };
                const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = r0 + e;
                    const float4 &acc = e ? acc1 : acc0;
                    put4(sm.tp, 8192, r, col,
                         scaled(*reinterpret_cast<const float4 *>(T1 + r * LDT + col), bl, 1.f));
                    put4(sm.tp, 8192, r, 32 + col, zero);
                    put4(sm.tp, 8192, 32 + r, col, scaled(acc, bl, -1.f));
                    put4(sm.tp, 8192, 32 + r, 32 + col,
                         scaled(*reinterpret_cast<const float4 *>(T2 + r * LDT + col), bh, 1.f));
                }
            }
        }
        publish_smem();

        // ---------------------------------------------- a6: U^T = (V^T - Z^T) T'^T
        if (tid == 0) {
            tc_fence_after();
            mma3_ts(tmem + kColZ, tmem + kColUb, desc_sw128(a_tp, 16, 1024), 512, 2, id_kk, false);
            mma_commit(smem_u32(&sm.bar_mma));
        }
        __syncwarp();
        mma_done();
        if (!top) {  // U^T -> bf16 pairs, the A operand of the next two products
            uint32_t x[32], hp[16], lp[16];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(tmem + lane_addr + kColZ + 32 * half, x);
                split_pairs(x, hp, lp);
                tmem_st16(tmem + lane_addr + kColUb + 16 * half, hp);
                tmem_st16(tmem + lane_addr + kColUb + 32 + 16 * half, lp);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        __syncthreads();

        // ---------------------------------------------- O^T += U^T M^T, S^T += U^T Kb
        if (tid == 0) {
            tc_fence_after();
            mma3_ts(tmem + kColO, tmem + kColUb, desc_sw128(a_mm, 16, 1024), 512, 2, id_kk, true);
            mma3_ts(tmem + kColS, tmem + kColUb, desc_sw128(a_kb, 8192, 1024), 512, 128, id_km, true);
            mma_commit(smem_u32(&sm.bar_mma));
        }
        __syncwarp();
        mma_done();
        if (!top) {
            const int vv = L - 64;
            uint32_t x[32];
            // output: lane 64 + v holds O^T[v][r]
            if (!no_out) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld32(tmem + lane_addr + kColO + 32 * half, x);
#pragma unroll 8
                    for (int j = 0; j < 32; ++j) {
                        const int r = 32 * half + j;
                        const size_t i = ((size_t)(t0 + r) * p.H + h) * D + vv;
                        if (r < valid && in_bounds(p.status, i, n_tok)) st(o, i, __uint_as_float(x[j]));
                    }
                }
            }
            // S^T <- (S^T + U^T Kb) Diag(gamma), and its bf16 pairs
            uint32_t hp[16], lp[16];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(tmem + lane_addr + kColS + 32 * half, x);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    x[c] = __float_as_uint(__uint_as_float(x[c]) * sm.gam[n & 1][32 * half + c]);
                tmem_st32(tmem + lane_addr + kColS + 32 * half, x);
                split_pairs(x, hp, lp);
                tmem_st16(tmem + lane_addr + kColSb + 16 * half, hp);
                tmem_st16(tmem + lane_addr + kColSb + 32 + 16 * half, lp);
            }
            tmem_wait_st();
        } else if (n + 1 < nchunks) {
            operands(n + 1);
        }
        publish_smem();
    }
    const bool domain = sm.domain;

    // final state: lane 64 + v holds row v of S^T
    if (!domain && !top && sref.S_T) {
        tc_fence_after();
        const int vv = L - 64;
        uint32_t x[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tmem_ld32(tmem + lane_addr + kColS + 32 * half, x);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const size_t i = sref.off + (size_t)vv * D + 32 * half + c;
                if (in_bounds(p.status, i, sref.ext)) sref.S_T[i] = __uint_as_float(x[c]);
            }
        }
    }
    // teardown: every MMA issued has completed before tensor memory is freed,
    // and the last row copy has landed (it is in flight only after a timeout)
    if (tid == 0) {
        mma_commit(smem_u32(&sm.bar_fin));
        wait_bounded(sm.bar_fin, 0);
        if (ld_issued > 0) wait_bounded(sm.bar_ld, (ld_issued - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && sm.abort) raise_status(p.status, KDA_ERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (domain && !sm.abort) serial_pass<T>(p, sm, start, len, h, sref);
}

// [Ttot][H][64] rows (fp32 or bf16) as a 3-D tensor, tile = 64 channels x one
// head x 64 tokens, unswizzled (the tile is dense in shared memory, row t at
// t * 64 elements); tokens past Ttot read as zero.
bool make_rows_map(CUtensorMap *map, const void *base, bool fp32, int H, int64_t Ttot) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    if (!enc) return false;
    const cuuint64_t eb = fp32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)Ttot};
    cuuint64_t strides[2] = {(cuuint64_t)D * eb, (cuuint64_t)H * D * eb};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)C};
    cuuint32_t elem[3] = {1, 1, 1};
    return enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_tc64(const FwdParams &p, kda_dtype_t dt, cudaStream_t s) {
    if ((size_t)p.N * p.H == 0) return cudaSuccess;
    if (p.Ttot > INT32_MAX || p.dk != D || p.dv != D) return cudaErrorInvalidValue;
    if (p.Ttot == 0) return launch_prefill_simt(p, dt, s);  // every sequence empty
    const bool f32 = dt == KDA_F32;
    CUtensorMap ml, mk, mq, mv;
    if (!make_rows_map(&ml, p.log_alpha, true, p.H, p.Ttot) ||
        !make_rows_map(&mk, p.k, f32, p.H, p.Ttot) || !make_rows_map(&mq, p.q, f32, p.H, p.Ttot) ||
        !make_rows_map(&mv, p.v, f32, p.H, p.Ttot))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(Tc64Smem) + 1024;
    const unsigned blocks = (unsigned)((size_t)p.N * p.H);
    auto kern = f32 ? prefill_tc64_kernel<float> : prefill_tc64_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<blocks, kThreads, smem, s>>>(p, ml, mk, mq, mv);
    return cudaGetLastError();
}

cudaError_t launch_prefill_tensorcore(const FwdParams &p, kda_dtype_t dt, cudaStream_t s) {
    return p.dk == D ? launch_prefill_tc64(p, dt, s) : launch_prefill_tc(p, s);
}

}  // namespace kda

// Tensor-core chunkwise KDA forward for d_k = d_v = 64 (fp32 or bf16 q/k/v,
// fp32 state) on sm_103a, to fp32 accuracy.
//
// The chunk form of the 128-wide engine ("Kimi Delta Attention 完全拆解",
// chunkwise section; "Kimi K3 的 KDA" section 5), every contraction on tcgen05:
//
//   G = in-chunk inclusive cumsum of log_alpha, Gamma = exp(G), gamma = Gamma_63
//   Kh = K . Gamma,  Qh = Q . Gamma,  Kb = K / Gamma
//   R = [Kh; Qh] Kb^T:  A = StrictTril(diag(beta) R_top),  M = Tril(R_bottom)
//   T' = (I + A)^-1 diag(beta)                      (fp32 forward substitution)
//   [W^T; U~^T] = [Kh^T; V^T] T'^T
//   U^T = U~^T - S^T W^T,  O^T = S^T Qh^T + U^T M^T,  S^T <- (S^T + U^T Kb) Diag(gamma)
//
// fp32 accuracy from the bf16 tensor cores: each operand x is held as the pair
// hi = bf16(x), lo = bf16(x - hi), which leaves x - hi - lo within 2^-17 |x|,
// and each product is the sum of hi.hi, hi.lo and lo.hi over K slices of 16,
// accumulated in fp32 in tensor memory (the dropped lo.lo term is ~2^-16 of
// the product).  A pair takes the bytes of one fp32 operand: the hi and lo tiles
// of a 64-wide head have the shape of the two 64-channel slabs of a 128-wide
// bf16 head and use the same 128-byte-swizzled layouts and descriptors.
//
// Every MMA has M = 128: R stacks the Kh and Qh rows, [W^T; U~^T] stacks the
// key and value features; the products whose left operand has 64 rows (S^T and
// U^T, bf16 pairs read from tensor memory) hold them in lanes 64-127, so their
// results land in lanes 64-127, and lanes 0-63 of those operands stay zero.
// So warps 0-1 (tensor-memory lanes 0-63) read out A and W^T, warps 2-3
// (lanes 64-127) M, U^T, O^T and the state.  One CTA of 128 threads per
// (sequence, head) walks the chunks one at a time; one thread issues the MMAs.
// A (sequence, head) with a chunk whose cumulative log-decay leaves [-80, 0]
// (exp(-G) past fp32 range) is recomputed token by token from S0 instead.
// Every mbarrier wait is bounded; a timeout records KDA_ERR_TIMEOUT.
#include <cuda.h>
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
constexpr uint32_t kColWU = 64;   // [W^T; U~^T], then lanes 64-127 U^T   (64 fp32)
constexpr uint32_t kColO = 128;   // O^T in lanes 64-127                  (64 fp32)
constexpr uint32_t kColS = 192;   // S^T master in lanes 64-127           (64 fp32)
constexpr uint32_t kColSb = 256;  // S^T bf16 pairs: hi 32 columns, lo 32 (A operand)
constexpr uint32_t kColUb = 320;  // U^T bf16 pairs: hi 32 columns, lo 32 (A operand)
constexpr int LDA = C + 1;        // fp32 row stride of the solve matrix

struct __align__(1024) Tc64Smem {
    uint8_t xq[32768];  // [Kh; Qh] K-major, 128 rows x 64 channels: hi tile | lo tile
    uint8_t kb[16384];  // Kb [j][c]: hi | lo; K-major B of R, MN-major B of the S update
    uint8_t kv[32768];  // [Kh | V] MN-major A of [W^T; U~^T]: per part (hi | lo) the
                        // key block [j][c] then the value block [j][v] (8 KB each)
    uint8_t tp[16384];  // T' [r][j] K-major: hi | lo
    uint8_t wn[16384];  // -W as [c][r] (MN-major B of U): hi | lo
    uint8_t mm[16384];  // M [r][j] K-major: hi | lo
    uint8_t raw[4 * C * 256];  // the next chunk's rows as they are in memory (cp.async):
                               // log_alpha, k, q, v, 64 rows each of 64 elements
    float a[C * LDA];   // beta-scaled A (fp32); staging of the token-by-token pass
    float gam[D];
    float bet[C];
    float rbet[C];      // the next chunk's beta
    uint64_t bar_mma, bar_fin;
    uint32_t tmem_base;
    int abort;
    int domain;
};

// Wait for a phase within the time limit, whatever the abort flag says (the
// teardown's wait for the last MMAs).
__device__ __forceinline__ void wait_bounded(uint64_t &bar, uint32_t parity) {
    if (mbar_try_wait(smem_u32(&bar), parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&bar), parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
}

// Global -> shared copies that complete asynchronously (cp.async; waited for
// with cp_async_wait_all before a barrier).
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// byte offset of element (row, col) of a 64-column tile part (128-byte rows)
__device__ __forceinline__ uint32_t at(int row, int col) { return sw128_offset(row, col); }

__device__ __forceinline__ void split(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));  // x - hi is exact in fp32
}

// element (row, col) of a hi / lo tile pair whose lo part starts `part` bytes on
__device__ __forceinline__ void put(uint8_t *tile, uint32_t part, int row, int col, float x) {
    __nv_bfloat16 hi, lo;
    split(x, hi, lo);
    *reinterpret_cast<__nv_bfloat16 *>(tile + at(row, col)) = hi;
    *reinterpret_cast<__nv_bfloat16 *>(tile + part + at(row, col)) = lo;
}

// columns col .. col + 7 (col a multiple of 8) of one row of a tile pair
__device__ __forceinline__ void put8(uint8_t *tile, uint32_t part, int row, int col,
                                     const float *x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat16 h0, l0, h1, l1;
        split(x[2 * i], h0, l0);
        split(x[2 * i + 1], h1, l1);
        h[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        l[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    *reinterpret_cast<uint4 *>(tile + at(row, col)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(tile + part + at(row, col)) = make_uint4(l[0], l[1], l[2], l[3]);
}

// 32 fp32 values of a tensor-memory row -> 16 hi pairs and 16 lo pairs (the
// even K index in the low half), the A-operand format of the MMA
__device__ __forceinline__ void split_pairs(const uint32_t (&x)[32], uint32_t (&h)[16],
                                            uint32_t (&l)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        __nv_bfloat16 h0, l0, h1, l1;
        split(__uint_as_float(x[2 * i]), h0, l0);
        split(__uint_as_float(x[2 * i + 1]), h1, l1);
        h[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        l[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
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
__global__ void __launch_bounds__(kThreads, 1) prefill_tc64_kernel(const __grid_constant__ FwdParams p) {
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
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    T *o = static_cast<T *>(p.o);

    volatile int *abort = &sm.abort;
    if (tid == 0) {
        sm.abort = 0;
        sm.domain = 0;
        mbar_init(smem_u32(&sm.bar_mma), 1);
        mbar_init(smem_u32(&sm.bar_fin), 1);
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

    const uint32_t a_xq = smem_u32(sm.xq), a_kb = smem_u32(sm.kb), a_kv = smem_u32(sm.kv);
    const uint32_t a_tp = smem_u32(sm.tp), a_wn = smem_u32(sm.wn), a_mm = smem_u32(sm.mm);
    const uint32_t id_kk = idesc_bf16(128, 64, false, false);  // K-major A and B
    const uint32_t id_mk = idesc_bf16(128, 64, true, false);   // MN-major A
    const uint32_t id_km = idesc_bf16(128, 64, false, true);   // MN-major B

    // chunk m's rows of log_alpha, k, q, v and its beta -> sm.raw / sm.rbet (all
    // threads, 16-byte copies; rows past the sequence end are not copied)
    constexpr int kRow = D * (int)sizeof(T);  // bytes of one k / q / v row
    float *raw_la = reinterpret_cast<float *>(sm.raw);
    const T *raw_k = reinterpret_cast<const T *>(sm.raw + C * 256);
    const T *raw_q = reinterpret_cast<const T *>(sm.raw + 2 * C * 256);
    const T *raw_v = reinterpret_cast<const T *>(sm.raw + 3 * C * 256);
    auto prefetch = [&](int m) {
        const int64_t tm = start + (int64_t)m * C;
        const int vm = min(C, len - m * C);
        for (int i = tid; i < vm * 16; i += kThreads) {  // log_alpha: 16 pieces per row
            const int t = i >> 4, c4 = (i & 15) * 4;
            const size_t g = ((size_t)(tm + t) * p.H + h) * D + c4;
            if (in_bounds(p.status, g + 3, n_tok)) cp_async16(raw_la + t * D + c4, p.log_alpha + g);
        }
        constexpr int kPieces = kRow / 16;
        for (int i = tid; i < 3 * vm * kPieces; i += kThreads) {
            const int w = i / (vm * kPieces), r = i % (vm * kPieces);
            const int t = r / kPieces, e = (r % kPieces) * (16 / (int)sizeof(T));
            if (w == 2 && vzero) continue;
            const T *src = w == 0 ? k : w == 1 ? q : v;
            const size_t g = ((size_t)(tm + t) * p.H + h) * D + e;
            if (in_bounds(p.status, g + 16 / sizeof(T) - 1, n_tok))
                cp_async16(sm.raw + (w + 1) * C * 256 + t * kRow + e * sizeof(T), src + g);
        }
        if (tid < vm) {
            const size_t bi = (size_t)(tm + tid) * p.H + h;
            if (in_bounds(p.status, bi, n_beta)) cp_async4(&sm.rbet[tid], p.beta + bi);
        }
    };
    prefetch(0);
    cp_async_wait_all();
    __syncthreads();

    for (int n = 0; n < nchunks; ++n) {
        const int64_t t0 = start + (int64_t)n * C;
        const int valid = min(C, len - n * C);
        // ---------------------------------------------- a1, a2: gates and operands
        // from the staged rows: thread (half, c) takes channel c of tokens
        // 32 half .. 32 half + 31 -- its k, q, v and gates; the second half
        // first sums the first half's log-decays for its starting G -- and
        // thread t < 64 the beta of token t
        {
            const int c = tid & (D - 1), half = tid >> 6;
            const int t_begin = 32 * half;
            float G = 0.f;
            if (half) {
#pragma unroll 8
                for (int t = 0; t < 32; ++t) G += t < valid ? raw_la[t * D + c] : 0.f;
            }
#pragma unroll 4
            for (int t = t_begin; t < t_begin + 32; ++t) {
                const bool live = t < valid;
                G += live ? raw_la[t * D + c] : 0.f;
                const float kf = live ? ld(raw_k, t * D + c) : 0.f;
                const float qf = live ? ld(raw_q, t * D + c) : 0.f;
                const float gf = expf(G), gi = expf(-G);
                const float kh = kf * gf;
                put(sm.xq, 16384, t, c, kh);
                put(sm.xq, 16384, 64 + t, c, qf * gf);
                put(sm.kb, 8192, t, c, kf * gi);
                put(sm.kv, 16384, t, c, kh);
                put(sm.kv + 8192, 16384, t, c, live && !vzero ? ld(raw_v, t * D + c) : 0.f);
                if (t == C - 1) sm.gam[c] = gf;
            }
            if (half && !(G >= -kLogDecayLimit)) *reinterpret_cast<volatile int *>(&sm.domain) = 1;
            if (tid < C) sm.bet[tid] = tid < valid ? sm.rbet[tid] : 0.f;
        }
        publish_smem();
        if (*reinterpret_cast<volatile int *>(&sm.domain)) break;  // (read by all after the barrier)
        if (n + 1 < nchunks) prefetch(n + 1);  // the staged rows have been read

        // ---------------------------------------------- a3, a5: R = [Kh; Qh] Kb^T
        if (tid == 0) {
            tc_fence_after();
            mma3_ss(tmem + kColR, desc_sw128(a_xq, 16, 1024), 1024, 2, desc_sw128(a_kb, 16, 1024),
                    512, 2, id_kk, false);
            mma_commit(smem_u32(&sm.bar_mma));
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
                    for (int j = 0; j < 32; ++j) sm.a[L * LDA + 32 * half + j] = br * __uint_as_float(x[j]);
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
        // thread j < 64: column j of T = (I + A)^-1 by forward substitution
        // (T[r][j] = -sum_{s < r} A[r][s] T[s][j] below the diagonal), two
        // partial sums to halve the dependency chain; then T'[r][j] = T[r][j] beta_j
        if (tid < C) {
            const int j = tid;
            float x[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int s = 0; s + 1 < r; s += 2) {
                    s0 = fmaf(sm.a[r * LDA + s], x[s], s0);
                    s1 = fmaf(sm.a[r * LDA + s + 1], x[s + 1], s1);
                }
                if (r & 1) s0 = fmaf(sm.a[r * LDA + r - 1], x[r - 1], s0);
                x[r] = r < j ? 0.f : r == j ? 1.f : -(s0 + s1);
            }
            const float bj = sm.bet[j];
#pragma unroll
            for (int r = 0; r < C; ++r) put(sm.tp, 8192, r, j, x[r] * bj);
        }
        publish_smem();

        // ---------------------------------------------- [W^T; U~^T] = [Kh^T; V^T] T'^T
        if (tid == 0) {
            tc_fence_after();
            mma3_ss(tmem + kColWU, desc_sw128(a_kv, 8192, 1024), 1024, 128,
                    desc_sw128(a_tp, 16, 1024), 512, 2, id_mk, false);
            mma_commit(smem_u32(&sm.bar_mma));
        }
        __syncwarp();
        mma_done();
        if (top) {  // -W as [c][r]: lane c holds row c of W^T
            uint32_t x[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(tmem + lane_addr + kColWU + 32 * half, x);
#pragma unroll
                for (int j8 = 0; j8 < 32; j8 += 8) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = -__uint_as_float(x[j8 + e]);
                    put8(sm.wn, 8192, L, 32 * half + j8, f);
                }
            }
        }
        publish_smem();

        // ---------------------------------------------- a6: U^T = U~^T - S^T W^T, O^T = S^T Qh^T
        if (tid == 0) {
            tc_fence_after();
            mma3_ts(tmem + kColWU, tmem + kColSb, desc_sw128(a_wn, 8192, 1024), 512, 128, id_km,
                    true);
            mma3_ts(tmem + kColO, tmem + kColSb, desc_sw128(a_xq + 8192, 16, 1024), 1024, 2, id_kk,
                    false);
            mma_commit(smem_u32(&sm.bar_mma));
        }
        __syncwarp();
        mma_done();
        if (!top) {  // U^T -> bf16 pairs, the A operand of the next two products
            uint32_t x[32], hp[16], lp[16];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld32(tmem + lane_addr + kColWU + 32 * half, x);
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
                for (int c = 0; c < 32; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) * sm.gam[32 * half + c]);
                tmem_st32(tmem + lane_addr + kColS + 32 * half, x);
                split_pairs(x, hp, lp);
                tmem_st16(tmem + lane_addr + kColSb + 16 * half, hp);
                tmem_st16(tmem + lane_addr + kColSb + 32 + 16 * half, lp);
            }
            tmem_wait_st();
        }
        cp_async_wait_all();  // the next chunk's rows have landed
        tc_fence_before();
        __syncthreads();
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
    // teardown: every MMA issued has completed before tensor memory is freed
    if (tid == 0) {
        mma_commit(smem_u32(&sm.bar_fin));
        wait_bounded(sm.bar_fin, 0);
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

}  // namespace

cudaError_t launch_prefill_tc64(const FwdParams &p, kda_dtype_t dt, cudaStream_t s) {
    if ((size_t)p.N * p.H == 0) return cudaSuccess;
    if (p.Ttot > INT32_MAX || p.dk != D || p.dv != D) return cudaErrorInvalidValue;
    const size_t smem = sizeof(Tc64Smem) + 1024;
    const unsigned blocks = (unsigned)((size_t)p.N * p.H);
    auto kern = dt == KDA_F32 ? prefill_tc64_kernel<float> : prefill_tc64_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<blocks, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_tensorcore(const FwdParams &p, kda_dtype_t dt, cudaStream_t s) {
    return p.dk == D ? launch_prefill_tc64(p, dt, s) : launch_prefill_tc(p, s);
}

}  // namespace kda

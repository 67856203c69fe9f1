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
// Every value channel (a row s of the [d_v][d_k] state) runs through the
// decode recurrence on its own ("Kimi Delta Attention 完全拆解", the KDA
// recurrence): s <- alpha_t * s; u_t = beta_t (v_t - s . k_t); s <- s + u_t k_t;
// o_t = s . q_t.  The tokens are taken in sub-blocks of up to 8, and within a
// sub-block the recurrence is unrolled in closed form -- the chunkwise algebra
// of the same page, for one chunk of <= 8 tokens seen from one row.  With
// D(j, t) = prod_{i = j+1 .. t} alpha_i (per key channel; D(t, t) = 1) and s
// the row entering the sub-block:
//
//   u_t = beta_t (v_t - s . (D(-1, t) k_t) - sum_{j<t} A[t][j] u_j),
//         A[t][j] = sum_c k_t[c] k_j[c] D(j, t)[c]
//   o_t = s . (D(-1, t) q_t) + sum_{j<=t} M[t][j] u_j,
//         M[t][j] = sum_c q_t[c] k_j[c] D(j, t)[c]
//   s'  = D(-1, n-1) s + sum_j u_j D(j, n-1) k_j
//
// The decays are running products of alpha (never exp of a difference of
// sums), so nothing overflows however strong the decay.  A, M and the decayed
// keys and queries belong to the (session, head) pair and are built once; per
// row the work is 2 n dot products of length d_k (n for commit), an n x n
// triangular solve and, for commit, an n-term update.
//
// Layout: one block of 2 d threads per (session, head) pair at a time (a grid
// of the resident blocks walks the pairs; while a pair is worked on, the next
// pair's state and first 8 token rows land in shared memory by cp.async).  Warp w owns state rows 16 w .. 16 w + 15, held in registers in
// the accumulator layout of an m16n8 tensor-core tile (lane (g, t): rows g and
// g + 8, key channels 8 i + 2 t and 8 i + 2 t + 1 of every 8-channel slice
// i).  Read with the k index of each slice taken in the order 2 t, 2 t + 1
// instead of t, t + 4, the same registers are the A fragments of m16n8k8
// products, so the 2 n dot products of a row are tensor-core products of the
// state with the decayed keys and queries -- fp32 accuracy from three tf32
// products per tile (high x high, high x low, low x high), except in a bf16
// verify, which only reads the state and rounds its outputs to bf16: bf16
// products there (m16n8k16, whose A fragment is the same registers taken 16
// channels at a time).  The solve and the
// state update stay in fp32 on the CUDA cores (the update adds into the same
// registers, round to nearest).
#include <cuda_bf16.h>

#include <atomic>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kSub = 8;  // draft tokens per sub-block

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// 2^x by the MUFU ex2 (about 2 ulp; alpha = 2^(log_alpha log2 e))
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x rounded to the nearest tf32 value (ties away from zero), as its fp32 bit
// pattern: add half a unit of the 13 dropped bits, then drop them (two integer
// instructions; a carry into the exponent is the correct rounding up)
__device__ __forceinline__ uint32_t tf32_bits(float x) {
    return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
}

// x = hi + lo, hi the nearest tf32 value (its low part, below tf32 resolution
// itself, is truncated by the tensor core: an error of 2^-11 of 2^-11 of x)
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = tf32_bits(x);
    lo = __float_as_uint(x - __uint_as_float(hi));
}

// bf16 pair {lo, hi} (lo in the low half), rounded to nearest
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// d (16 x 8, fp32) += a (16 x 16) b (16 x 8), bf16 operands
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d (16 x 8, fp32) += a (16 x 8) b (8 x 8), tf32 operands
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d[0] + d[1] + d[2] += a b to fp32 accuracy from the split operands: low x
// high, high x low and high x high into three accumulators (three independent
// chains; the low x low product is below fp32 resolution and left out)
__device__ __forceinline__ void mma_3xtf32(float (&d)[3][4], const uint32_t (&ah)[4],
                                           const uint32_t (&al)[4], float2 bh, float2 bl) {
    mma_tf32(d[0], al, __float_as_uint(bh.x), __float_as_uint(bh.y));
    mma_tf32(d[1], ah, __float_as_uint(bl.x), __float_as_uint(bl.y));
    mma_tf32(d[2], ah, __float_as_uint(bh.x), __float_as_uint(bh.y));
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16 bytes global -> shared, asynchronously (cp.async, completion per thread)
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Sum of x over the kLen lanes whose indices differ only in the bits below
// kLen (a halving butterfly: kLen - 1 shuffles for kLen values).  Lane l is
// left with the total of x[l % kLen].
template <int kLen>
__device__ __forceinline__ float halving_sum(float (&x)[kLen], int lane) {
#pragma unroll
    for (int len = kLen / 2; len >= 1; len >>= 1) {
        const bool up = lane & len;
#pragma unroll
        for (int i = 0; i < len; ++i) {
            const float keep = up ? x[i + len] : x[i];
            const float send = up ? x[i] : x[i + len];
            x[i] = keep + __shfl_xor_sync(0xffffffffu, send, len);
        }
    }
    return x[0];
}

template <int D, typename Tin>
struct DraftSmem {
    static constexpr int kLd = D + 8;  // padded rows: conflict-free fragment loads
    // tensor-core operands as a tf32 high part [0] and the rest [1] (a bf16
    // verify keeps its bf16 keys and queries in [1], rows of D + 8 elements)
    float xk[2][kSub][kLd];  // D(-1, t) k_t
    float xq[2][kSub][kLd];  // D(-1, t) q_t
    float kb[2][kSub][kLd];  // D(t, n-1) k_t
    float vs[kSub][D];       // v_t
    float gam[D];            // D(-1, n-1)
    float beta[kSub];
    float A[kSub][kSub];  // strictly lower
    float M[kSub][kSub];  // lower, with the diagonal
    float part[2][D / 32][32];
    // the token rows of the next pair's first sub-block, landed by cp.async
    Tin tk[kSub][D], tq[kSub][D], tv[kSub][D];
    float tl[kSub][D];
};

// Entries of one of the two partial-sum sets: index t (t - 1) / 2 + j < 28 is
// the strictly lower entry (t, j); 28 .. 31 are diagonal entries.
__device__ __forceinline__ void lower_entry(int l, int &t, int &j) {
    t = 1;
    while (t * (t + 1) / 2 <= l) ++t;
    j = l - t * (t - 1) / 2;
}

// x[j] and x[j + 4] for a lane-dependent j in 0 .. 3 (registers take no
// runtime index)
__device__ __forceinline__ float pick4(const float (&x)[kSub], int j, int off) {
    const float lo = j & 1 ? x[off + 1] : x[off];
    const float hi = j & 1 ? x[off + 3] : x[off + 2];
    return j & 2 ? hi : lo;
}

template <int D, typename Tin, bool kCommit>
__global__ void __launch_bounds__(2 * D, 2) draft_kernel(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
    const float *__restrict__ log_alpha, const float *__restrict__ beta, float *__restrict__ S,
    const int32_t *__restrict__ n_accept, Tin *__restrict__ o, int N, int K, int H,
    int tokens_aligned) {
    constexpr int kNT = D / 8;  // 8-channel slices of a row
    constexpr int kThreads = 2 * D;
    // verify with bf16 outputs (the state only read): the dots are bf16
    // products (state rows and decayed keys / queries rounded to bf16, as the
    // tensor-core prefill reads its state), under the outputs' own bf16
    // rounding.  Everything that updates the state keeps the three-product
    // fp32 form.
    constexpr bool kBf16Dots = !kCommit && sizeof(Tin) == 2;
    constexpr int kLdb = D + 8;  // bf16 operand rows, over the (then unused) low-part arrays
    extern __shared__ __align__(16) uint8_t draft_smem[];
    DraftSmem<D, Tin> &sm = *reinterpret_cast<DraftSmem<D, Tin> *>(draft_smem);
    // the next pair's state, landed by cp.async while this pair is worked on;
    // 16-byte chunk j of row r sits at chunk j ^ (r % 8) (conflict-free reads)
    float *st = reinterpret_cast<float *>(draft_smem + sizeof(DraftSmem<D, Tin>));

    const int tid = threadIdx.x, lane = tid & 31;
    // set-up roles: key / value channel c, and which half of the work
    const int c = tid % D, half = tid / D;
    // row roles: fragment rows rA, rB = rA + 8 (lane (g, tg) of warp w); the
    // lane solves row rA (tg < 2) or rB and writes the tokens of parity tg % 2
    const int g = lane >> 2, tg = lane & 3;
    const int rA = 16 * (tid >> 5) + g, rB = rA + 8;
    const int rsel = tg >> 1, par = tg & 1;
    const int myrow = rsel ? rB : rA;
    const int NH = N * H;

    // State and first-sub-block token rows of pair pp into shared memory.  A
    // thread copies the same chunks every time, so its own wait orders each
    // copy after the one before it.
    auto stage = [&](int pp) {
        if (pp >= NH) return;
        const float *src = S + (size_t)pp * D * D;
        for (int i = tid; i < D * D / 4; i += kThreads) {
            const int r = i / (D / 4), j = i % (D / 4);
            cp_async16(st + r * D + 4 * (j ^ (r & 7)), src + r * D + 4 * j);
        }
        const int n2 = pp / H, h2 = pp % H, nt = min(K, kSub);
        auto row = [&](int t) { return ((size_t)(n2 * K + t) * H + h2) * D; };
        if (tokens_aligned) {
            constexpr int kPer = 16 / sizeof(Tin);  // elements per 16-byte chunk
            for (int i = tid; i < nt * (D / kPer); i += kThreads) {
                const int t = i / (D / kPer), e = (i % (D / kPer)) * kPer;
                cp_async16(&sm.tk[t][e], k + row(t) + e);
                cp_async16(&sm.tv[t][e], v + row(t) + e);
                if (!kCommit) cp_async16(&sm.tq[t][e], q + row(t) + e);
            }
            for (int i = tid; i < nt * (D / 4); i += kThreads) {
                const int t = i / (D / 4), e = (i % (D / 4)) * 4;
                cp_async16(&sm.tl[t][e], log_alpha + row(t) + e);
            }
        } else {
            for (int i = tid; i < nt * D; i += kThreads) {
                const int t = i / D, e = i % D;
                sm.tk[t][e] = k[row(t) + e];
                sm.tv[t][e] = v[row(t) + e];
                if (!kCommit) sm.tq[t][e] = q[row(t) + e];
                sm.tl[t][e] = log_alpha[row(t) + e];
            }
        }
        cp_async_commit();
    };
    stage(blockIdx.x);

    for (int p = blockIdx.x; p < NH; p += gridDim.x) {
        const int n = p / H, h = p % H;
        const int ntok = kCommit && n_accept ? min(max(n_accept[n], 0), K) : K;
        cp_async_wait_all();
        if (ntok == 0) {  // nothing accepted: S stays as it is
            stage(p + gridDim.x);
            continue;
        }
        float *Sp = S + (size_t)p * D * D;
        float2 sa[kNT], sb[kNT];  // rows rA, rB; channels 8 i + 2 tg, + 1

        for (int t0 = 0; t0 < ntok; t0 += kSub) {
            const int nb = min(kSub, ntok - t0);
            const bool update = kCommit || t0 + kSub < ntok;
            __syncthreads();  // staged rows landed; the last sub-block is done with smem

            // ---- per-pair set-up: decayed keys / queries, A and M partial sums
            float a[kSub], kk[kSub], qq[kSub];
#pragma unroll
            for (int t = 0; t < kSub; ++t) {
                const bool live = t < nb;
                float la = 0.f, kv = 0.f, qv = 0.f;
                if (t0 == 0) {  // staged
                    la = sm.tl[t][c];
                    kv = to_f(sm.tk[t][c]);
                    if (!kCommit) qv = to_f(sm.tq[t][c]);
                } else if (live) {  // later sub-blocks read global memory
                    const size_t gi = ((size_t)(n * K + t0 + t) * H + h) * D + c;
                    la = log_alpha[gi];
                    kv = to_f(k[gi]);
                    if (!kCommit) qv = to_f(q[gi]);
                }
                a[t] = live ? ex2_fast(la * 1.4426950408889634f) : 1.f;
                kk[t] = live ? kv : 0.f;
                qq[t] = live ? qv : 0.f;
            }
            if (half == 0) {
                float run = 1.f;
#pragma unroll
                for (int t = 0; t < kSub; ++t) {
                    run *= a[t];
                    if constexpr (kBf16Dots) {
                        reinterpret_cast<__nv_bfloat16 *>(&sm.xk[1][0][0])[t * kLdb + c] =
                            __float2bfloat16_rn(kk[t] * run);
                    } else {
                        uint32_t hi, lo;
                        split_tf32(kk[t] * run, hi, lo);
                        sm.xk[0][t][c] = __uint_as_float(hi);
                        sm.xk[1][t][c] = __uint_as_float(lo);
                    }
                }
            } else {
                float run = 1.f;
#pragma unroll
                for (int t = 0; t < kSub; ++t) {
                    run *= a[t];
                    if (!kCommit) {
                        if constexpr (kBf16Dots) {
                            reinterpret_cast<__nv_bfloat16 *>(&sm.xq[1][0][0])[t * kLdb + c] =
                                __float2bfloat16_rn(qq[t] * run);
                        } else {
                            uint32_t hi, lo;
                            split_tf32(qq[t] * run, hi, lo);
                            sm.xq[0][t][c] = __uint_as_float(hi);
                            sm.xq[1][t][c] = __uint_as_float(lo);
                        }
                    }
                }
                if (update) {
                    sm.gam[c] = run;
                    float tail = 1.f;
#pragma unroll
                    for (int t = kSub - 1; t >= 0; --t) {
                        uint32_t hi, lo;
                        split_tf32(kk[t] * tail, hi, lo);
                        sm.kb[0][t][c] = __uint_as_float(hi);
                        sm.kb[1][t][c] = __uint_as_float(lo);
                        tail *= a[t];
                    }
                }
#pragma unroll
                for (int t = 0; t < kSub; ++t) {
                    float vv = 0.f;
                    if (t < nb)
                        vv = t0 == 0 ? to_f(sm.tv[t][c])
                                     : to_f(v[((size_t)(n * K + t0 + t) * H + h) * D + c]);
                    sm.vs[t][c] = vv;
                }
            }
            if (tid < kSub)
                sm.beta[tid] = tid < nb ? beta[(size_t)(n * K + t0 + tid) * H + h] : 0.f;
            if constexpr (kCommit) {
                // commit needs A alone: its 28 entries split by rows between the
                // halves (rows 1-5, 15 entries, on half 0; rows 6-7, 13, on half 1)
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = 0.f;
                if (half == 0) {
#pragma unroll
                    for (int t = 1; t <= 5; ++t) {
                        float dec = 1.f;
#pragma unroll
                        for (int j = t - 1; j >= 0; --j) {
                            dec *= a[j + 1];
                            x[t * (t - 1) / 2 + j] = kk[t] * kk[j] * dec;
                        }
                    }
                } else {
#pragma unroll
                    for (int t = 6; t < kSub; ++t) {
                        float dec = 1.f;
#pragma unroll
                        for (int j = t - 1; j >= 0; --j) {
                            dec *= a[j + 1];
                            x[t * (t - 1) / 2 + j - 15] = kk[t] * kk[j] * dec;
                        }
                    }
                }
                float sum16 = halving_sum<16>(x, lane);  // over this half-warp
                sum16 += __shfl_xor_sync(0xffffffffu, sum16, 16);
                sm.part[half][c >> 5][lane] = sum16;
            } else {
                // half 0: A[t][j] and M[t][t] for t < 4; half 1: M[t][j] (j < t)
                // and M[t][t] for t >= 4 -- this channel's terms
                float x[32];
#pragma unroll
                for (int t = 1; t < kSub; ++t) {
                    const float lhs = half == 0 ? kk[t] : qq[t];
                    float dec = 1.f;
#pragma unroll
                    for (int j = t - 1; j >= 0; --j) {
                        dec *= a[j + 1];
                        x[t * (t - 1) / 2 + j] = lhs * kk[j] * dec;
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    x[28 + t] = half == 0 ? qq[t] * kk[t] : qq[t + 4] * kk[t + 4];
                sm.part[half][c >> 5][lane] = halving_sum<32>(x, lane);
            }
            __syncthreads();
            if (kCommit && tid < 28) {
                const int hh = tid < 15 ? 0 : 1, l = tid < 15 ? tid : tid - 15;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < D / 32; ++w) sum += sm.part[hh][w][l];
                int t, j;
                lower_entry(tid, t, j);
                sm.A[t][j] = sum;
            } else if (!kCommit && tid < 64) {
                const int hh = tid >> 5, l = tid & 31;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < D / 32; ++w) sum += sm.part[hh][w][l];
                if (l < 28) {
                    int t, j;
                    lower_entry(l, t, j);
                    if (hh == 0)
                        sm.A[t][j] = sum;
                    else
                        sm.M[t][j] = sum;
                } else {
                    const int t = l - 28 + 4 * hh;
                    sm.M[t][t] = sum;
                }
            }
            if (t0 == 0) {
#pragma unroll
                for (int i = 0; i < kNT; ++i) {
                    const int sw = 4 * ((2 * i + (tg >> 1)) ^ (rA & 7)) + 2 * (tg & 1);
                    sa[i] = *reinterpret_cast<const float2 *>(st + rA * D + sw);
                    sb[i] = *reinterpret_cast<const float2 *>(st + rB * D + sw);
                }
            }
            __syncthreads();  // A and M in place; the staged state and rows are read
            if (t0 == 0) stage(p + gridDim.x);

            // ---- per row: dot products with the decayed keys and queries on the
            // tensor cores.  Slice i is k step i; k index j < 4 is channel
            // 8 i + 2 j, j >= 4 is 8 i + 2 (j - 4) + 1, for the state (A) and the
            // keys / queries (B) alike.
            float cp3[3][4] = {}, cq3[3][4] = {};
            if constexpr (kBf16Dots) {
                // bf16 products, 16 channels per step: lane (g, tg) holds channels
                // 16 j + 2 tg, + 1 (slice 2 j) and 16 j + 8 + 2 tg, + 1 (slice 2 j + 1)
                const __nv_bfloat16 *xkb = reinterpret_cast<const __nv_bfloat16 *>(&sm.xk[1][0][0]);
                const __nv_bfloat16 *xqb = reinterpret_cast<const __nv_bfloat16 *>(&sm.xq[1][0][0]);
#pragma unroll
                for (int j = 0; j < kNT / 2; ++j) {
                    const uint32_t a[4] = {pack_bf16x2(sa[2 * j].x, sa[2 * j].y),
                                           pack_bf16x2(sb[2 * j].x, sb[2 * j].y),
                                           pack_bf16x2(sa[2 * j + 1].x, sa[2 * j + 1].y),
                                           pack_bf16x2(sb[2 * j + 1].x, sb[2 * j + 1].y)};
                    const int e = g * kLdb + 16 * j + 2 * tg;
                    mma_bf16(cp3[j % 3], a, *reinterpret_cast<const uint32_t *>(xkb + e),
                             *reinterpret_cast<const uint32_t *>(xkb + e + 8));
                    mma_bf16(cq3[j % 3], a, *reinterpret_cast<const uint32_t *>(xqb + e),
                             *reinterpret_cast<const uint32_t *>(xqb + e + 8));
                }
            } else {
#pragma unroll
                for (int i = 0; i < kNT; ++i) {
                    const int col = 8 * i + 2 * tg;  // B fragment: token g, channels col, col + 1
                    uint32_t ah[4], al[4];
                    split_tf32(sa[i].x, ah[0], al[0]);
                    split_tf32(sb[i].x, ah[1], al[1]);
                    split_tf32(sa[i].y, ah[2], al[2]);
                    split_tf32(sb[i].y, ah[3], al[3]);
                    mma_3xtf32(cp3, ah, al, *reinterpret_cast<const float2 *>(&sm.xk[0][g][col]),
                               *reinterpret_cast<const float2 *>(&sm.xk[1][g][col]));
                    if (!kCommit)
                        mma_3xtf32(cq3, ah, al,
                                   *reinterpret_cast<const float2 *>(&sm.xq[0][g][col]),
                                   *reinterpret_cast<const float2 *>(&sm.xq[1][g][col]));
                }
            }
            float cp[4], cq[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                cp[e] = (cp3[0][e] + cp3[1][e]) + cp3[2][e];
                cq[e] = (cq3[0][e] + cq3[1][e]) + cq3[2][e];
            }
            // cp: (rA, 2 tg), (rA, 2 tg + 1), (rB, 2 tg), (rB, 2 tg + 1); gather
            // the 8 tokens of the solved row from the 4 lanes of the quad
            float Pf[kSub], Qf[kSub];
            const int quad = lane & ~3;
#pragma unroll
            for (int src = 0; src < 4; ++src) {
                const float p0 = __shfl_sync(0xffffffffu, cp[0], quad + src);
                const float p1 = __shfl_sync(0xffffffffu, cp[1], quad + src);
                const float p2 = __shfl_sync(0xffffffffu, cp[2], quad + src);
                const float p3 = __shfl_sync(0xffffffffu, cp[3], quad + src);
                Pf[2 * src] = rsel ? p2 : p0;
                Pf[2 * src + 1] = rsel ? p3 : p1;
                if (!kCommit) {
                    const float q0 = __shfl_sync(0xffffffffu, cq[0], quad + src);
                    const float q1 = __shfl_sync(0xffffffffu, cq[1], quad + src);
                    const float q2 = __shfl_sync(0xffffffffu, cq[2], quad + src);
                    const float q3 = __shfl_sync(0xffffffffu, cq[3], quad + src);
                    Qf[2 * src] = rsel ? q2 : q0;
                    Qf[2 * src + 1] = rsel ? q3 : q1;
                }
            }
            // ---- triangular solve for u (tokens past nb have beta = 0: u = 0)
            float u[kSub];
#pragma unroll
            for (int t = 0; t < kSub; ++t) {
                float x = sm.vs[t][myrow] - Pf[t];
#pragma unroll
                for (int j = 0; j < t; ++j) x = fmaf(-sm.A[t][j], u[j], x);
                u[t] = sm.beta[t] * x;
            }
            if (!kCommit) {
#pragma unroll
                for (int t = 0; t < kSub; ++t) {
                    if (t < nb && (t & 1) == par) {
                        float ot = Qf[t];
#pragma unroll
                        for (int j = 0; j <= t; ++j) ot = fmaf(sm.M[t][j], u[j], ot);
                        o[((size_t)(n * K + t0 + t) * H + h) * D + myrow] = from_f<Tin>(ot);
                    }
                }
            }
            // ---- state update s <- D(-1, n-1) s + U Kb^T, the product on the
            // tensor cores (k = token) into a fresh accumulator, added in fp32
            if (update) {
                float ua[kSub], ub[kSub];  // u of rows rA and rB (lane tg ^ 2 solved the other)
#pragma unroll
                for (int t = 0; t < kSub; ++t) {
                    const float other = __shfl_xor_sync(0xffffffffu, u[t], 2);
                    ua[t] = rsel ? other : u[t];
                    ub[t] = rsel ? u[t] : other;
                }
                uint32_t uh[4], ul[4];  // A fragment: (rA, tg), (rB, tg), (rA, tg + 4), (rB, tg + 4)
                split_tf32(pick4(ua, tg, 0), uh[0], ul[0]);
                split_tf32(pick4(ub, tg, 0), uh[1], ul[1]);
                split_tf32(pick4(ua, tg, 4), uh[2], ul[2]);
                split_tf32(pick4(ub, tg, 4), uh[3], ul[3]);
#pragma unroll
                for (int i = 0; i < kNT; ++i) {
                    const int col = 8 * i + g;  // B fragment: tokens tg, tg + 4; channel col
                    const float2 bh = make_float2(sm.kb[0][tg][col], sm.kb[0][tg + 4][col]);
                    const float2 bl = make_float2(sm.kb[1][tg][col], sm.kb[1][tg + 4][col]);
                    float d3[3][4] = {};
                    mma_3xtf32(d3, uh, ul, bh, bl);
                    const float2 gm = *reinterpret_cast<const float2 *>(&sm.gam[8 * i + 2 * tg]);
                    sa[i].x = fmaf(gm.x, sa[i].x, (d3[0][0] + d3[1][0]) + d3[2][0]);
                    sa[i].y = fmaf(gm.y, sa[i].y, (d3[0][1] + d3[1][1]) + d3[2][1]);
                    sb[i].x = fmaf(gm.x, sb[i].x, (d3[0][2] + d3[1][2]) + d3[2][2]);
                    sb[i].y = fmaf(gm.y, sb[i].y, (d3[0][3] + d3[1][3]) + d3[2][3]);
                }
            }
        }
        if (kCommit) {
#pragma unroll
            for (int i = 0; i < kNT; ++i) {
                *reinterpret_cast<float2 *>(Sp + (size_t)rA * D + 8 * i + 2 * tg) = sa[i];
                *reinterpret_cast<float2 *>(Sp + (size_t)rB * D + 8 * i + 2 * tg) = sb[i];
            }
        }
    }
    cp_async_wait_all();  // nothing in flight at exit
}

template <int D, typename Tin, bool kCommit>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *la,
                         const float *beta, float *S, const int32_t *n_accept, void *o, int N,
                         int K, int H, cudaStream_t s) {
    constexpr int kMaxDevices = 64;
    // resident blocks per device (threads that race here all store the same value)
    static std::atomic<int> resident[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    constexpr size_t kSmem = sizeof(DraftSmem<D, Tin>) + (size_t)D * D * sizeof(float);
    int res = resident[dev].load(std::memory_order_relaxed);
    if (res == 0) {
        int sms = 0, per = 0;
        e = cudaFuncSetAttribute(draft_kernel<D, Tin, kCommit>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per, draft_kernel<D, Tin, kCommit>, 2 * D, kSmem);
        if (e != cudaSuccess) return e;
        res = sms * (per > 0 ? per : 1);
        resident[dev].store(res, std::memory_order_relaxed);
    }
    // token rows are staged by 16-byte copies when every row starts on 16 bytes
    const int pf = ((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)la) % 16 == 0;
    const int pairs = N * H;
    const int grid = pairs < res ? pairs : res;
    draft_kernel<D, Tin, kCommit><<<grid, 2 * D, kSmem, s>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        la, beta, S, n_accept, static_cast<Tin *>(o), N, K, H, pf);
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

// Chunkwise KDA forward on CUDA cores, all arithmetic in fp32.
//
// This engine serves fp32 inputs (whose tolerance needs fp32 arithmetic),
// d = 64, and any call that selects KDA_ENGINE_CUDACORE.  It runs the same
// chunk algorithm as the tensor-core engine, one 256-thread block per
// (sequence, head), all chunk tiles in shared memory:
//
//   per 64-token chunk, with G = in-chunk cumulative sum of log_alpha (inclusive),
//   Gamma = exp(G), gamma = Gamma at the chunk's last token:
//     Qh = Q . Gamma,  Kh = K . Gamma,  Kb = K / Gamma                 (a1, a2)
//     A  = StrictTril(diag(beta) Kh Kb^T)                              (a3)
//     (I + A) [W | U~] = diag(beta) [Kh | V]   (forward substitution)  (a4)
//     U  = U~ - W S                                                   (a6)
//     O  = Qh S + Tril(Qh Kb^T) U                                      (a5, a6)
//     S  <- Diag(gamma) (S + Kb^T U)                                   (a6)
//
// Derivation and sources.  Within a chunk, writing S_r = Diag(alpha_r) S_{r-1}
// + k_r u_r^T (u_r = beta_r (v_r - S̄_r^T k_r) is the delta-rule correction) and
// unrolling gives S_r = Diag(Gamma_r) [S + sum_{j<=r} Diag(1/Gamma_j) k_j u_j^T];
// reading that with k_r and q_r yields the triangular system for U and the
// output formula of "Kimi Delta Attention 完全拆解" (chunkwise section:
// O = (Gamma . Q) S + Tril[(Gamma . Q)(K / Gamma)^T](U - W S), and the state
// hand-off S <- Diag(gamma_C) S + (Gamma^{i->C} . K)^T (U - W S)).  The decay of
// a write at token i up to the chunk end is exp(G_C - G_i), i.e. gamma / Gamma_i,
// so the hand-off equals Diag(gamma) (S + Kb^T U).  The triangular solve is the
// UT transform those pages name; "Kimi K3 的 KDA" section 5 gives the same
// factorisation of the decay onto queries and keys.  The strict lower mask in
// the solve and the inclusive mask on the output (a token reads its own write)
// follow from the unrolled recurrence.
//
// Padding: a ragged tail chunk is filled with identity tokens (k = 0, v = 0,
// q = 0, log_alpha = 0, beta = 0), which leave S unchanged; their outputs are
// not stored.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_serial.cuh"

namespace kda {
namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <int D>
struct SimtSmem {
    static constexpr int LD = D + 1;      // odd row stride: conflict-free column walks
    static constexpr int LDA = C + 1;
    float Qh[C * LD];
    float Kh[C * LD];   // K . Gamma, then W
    float Kb[C * LD];   // log_alpha (phase 1 only), then K / Gamma
    float Vb[C * LD];   // V, then U~, then U
    float A[C * LDA];   // strict-lower solve matrix, then the output mask
    float S[D * LD];    // logical S[c][v], fp32
    float gam[D];
    float bet[C];
};

template <int D, typename Tin>
__global__ void __launch_bounds__(kThreads, 1) prefill_simt_kernel(FwdParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    using Sm = SimtSmem<D>;
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);
    constexpr int LD = Sm::LD, LDA = Sm::LDA;
    constexpr int NJ = D / 16;  // output columns per thread in 64 x D products

    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    if (*p.status == KDA_ERR_INVALID_ARGUMENT) return;  // set by the schedule kernel
    const int h = blockIdx.x % p.H;
    const int rank = blockIdx.x / p.H;
    const int n = p.order ? p.order[rank] : rank;

    int64_t start;
    int len;
    seq_range(p, n, start, len);
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    Tin *o = static_cast<Tin *>(p.o);
    const StateRef sref = state_ref(p, n, h, D, D);  // S0 / S_T block and task flags
    const bool vzero = sref.flags & kTaskVZero;
    if (sref.flags & kTaskNoOutput) o = nullptr;
    const size_t n_tok = (size_t)p.Ttot * p.H * D, n_beta = (size_t)p.Ttot * p.H;

    // initial state: memory [v][c] -> logical S[c][v]
    for (int idx = tid; idx < D * D; idx += kThreads) {
        const int vv = idx / D, c = idx % D;
        sm.S[c * LD + vv] =
            in_bounds(p.status, sref.off + idx, sref.ext) ? state_init(sref, vv, c, D) : 0.f;
    }

    const int nchunks = (len + C - 1) / C;
    for (int ch = 0; ch < nchunks; ++ch) {
        const int64_t t0 = start + (int64_t)ch * C;
        const int valid = min(C, len - ch * C);
        __syncthreads();  // previous chunk finished with every tile

        // ---- phase 1a: load the chunk (identity tokens past the end)
        for (int idx = tid; idx < C * D; idx += kThreads) {
            const int r = idx / D, c = idx % D;
            const size_t gi = ((size_t)(t0 + r) * p.H + h) * D + c;
            const bool ok = r < valid && in_bounds(p.status, gi, n_tok);
            sm.Qh[r * LD + c] = ok ? to_f(q[gi]) : 0.f;
            sm.Kh[r * LD + c] = ok ? to_f(k[gi]) : 0.f;
            sm.Vb[r * LD + c] = ok && !vzero ? to_f(v[gi]) : 0.f;
            sm.Kb[r * LD + c] = ok ? p.log_alpha[gi] : 0.f;
        }
        if (tid < C) {
            const size_t bi = (size_t)(t0 + tid) * p.H + h;
            sm.bet[tid] = tid < valid && in_bounds(p.status, bi, n_beta) ? p.beta[bi] : 0.f;
        }
        __syncthreads();

        // ---- a chunk whose cumulative log-decay leaves [-80, 80] in some
        // channel is taken token by token (exp(-G) would overflow fp32)
        bool wide = false;
        if (tid < D) {
            float G = 0.f;
            for (int r = 0; r < C; ++r) {
                G += sm.Kb[r * LD + tid];
                wide |= !(fabsf(G) <= kLogDecayLimit);
            }
        }
        if (__syncthreads_or(wide)) {
            for (int idx = tid; idx < valid * D; idx += kThreads) {
                const int r = idx / D, c = idx % D;
                sm.Kb[r * LD + c] = expf(sm.Kb[r * LD + c]);  // alpha
            }
            constexpr int CP = Serial<D>::kCP;
            const int vcol = tid % D, c0 = (tid / D) * CP;
            float st[CP];
#pragma unroll
            for (int i = 0; i < CP; ++i) st[i] = sm.S[(c0 + i) * LD + vcol];
            __syncthreads();
            // column sums in the (free) solve matrix: red_r then red_o
            serial_tokens<D, false, false>(st, sm.Kh, sm.Qh, sm.Kb, sm.Vb, sm.bet, LD, valid,
                                           sm.A, sm.A + 2 * Serial<D>::kParts * D, o,
                                           ((size_t)t0 * p.H + h) * D, (size_t)p.H * D, n_tok,
                                           p.status, 1);
#pragma unroll
            for (int i = 0; i < CP; ++i) sm.S[(c0 + i) * LD + vcol] = st[i];
            continue;
        }

        // ---- phase 1b: cumulative log-decay per key channel, scaled operands
        if (tid < D) {
            const int c = tid;
            float G = 0.f;
            for (int r = 0; r < C; ++r) {
                G += sm.Kb[r * LD + c];
                const float gf = expf(G), gi = expf(-G);
                const float kv = sm.Kh[r * LD + c];
                sm.Qh[r * LD + c] *= gf;
                sm.Kh[r * LD + c] = kv * gf;
                sm.Kb[r * LD + c] = kv * gi;
            }
            sm.gam[c] = expf(G);
        }
        __syncthreads();

        // ---- phase 2: A = StrictTril(diag(beta) Kh Kb^T)
        {
            float acc[4][4] = {};
            for (int c = 0; c < D; ++c) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = sm.Kh[(ty + 16 * i) * LD + c];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = sm.Kb[(tx + 16 * j) * LD + c];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = ty + 16 * i, jj = tx + 16 * j;
                    sm.A[r * LDA + jj] = jj < r ? sm.bet[r] * acc[i][j] : 0.f;
                }
        }
        __syncthreads();

        // ---- phase 3: forward substitution (I + A) X = diag(beta) [Kh | V],
        // one column of X per thread, written in place (W over Kh, U~ over V).
        if (tid < 2 * D) {
            float *col = tid < D ? sm.Kh + tid : sm.Vb + (tid - D);
            for (int r = 0; r < C; ++r) {
                float x = sm.bet[r] * col[r * LD];
                for (int j = 0; j < r; ++j) x = fmaf(-sm.A[r * LDA + j], col[j * LD], x);
                col[r * LD] = x;
            }
        }
        __syncthreads();

        // ---- phase 3b: output mask M = Tril(Qh Kb^T) (diagonal included), over A
        {
            float acc[4][4] = {};
            for (int c = 0; c < D; ++c) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = sm.Qh[(ty + 16 * i) * LD + c];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = sm.Kb[(tx + 16 * j) * LD + c];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = ty + 16 * i, jj = tx + 16 * j;
                    sm.A[r * LDA + jj] = jj <= r ? acc[i][j] : 0.f;
                }
        }

        // ---- phase 4: U = U~ - W S and the inter-chunk read Qh S
        float acc_o[4][NJ];
        {
            float acc_u[4][NJ];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < NJ; ++j) acc_u[i][j] = acc_o[i][j] = 0.f;
            for (int c = 0; c < D; ++c) {
                float w[4], qh[4], s[NJ];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w[i] = sm.Kh[(ty + 16 * i) * LD + c];
                    qh[i] = sm.Qh[(ty + 16 * i) * LD + c];
                }
#pragma unroll
                for (int j = 0; j < NJ; ++j) s[j] = sm.S[c * LD + tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        acc_u[i][j] = fmaf(w[i], s[j], acc_u[i][j]);
                        acc_o[i][j] = fmaf(qh[i], s[j], acc_o[i][j]);
                    }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    float &u = sm.Vb[(ty + 16 * i) * LD + tx + 16 * j];
                    u -= acc_u[i][j];
                }
        }
        __syncthreads();

        // ---- phase 5: O = Qh S + M U, stored for valid rows
        for (int jr = 0; jr < C; ++jr) {
            float u[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) u[j] = sm.Vb[jr * LD + tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float m = sm.A[(ty + 16 * i) * LDA + jr];
#pragma unroll
                for (int j = 0; j < NJ; ++j) acc_o[i][j] = fmaf(m, u[j], acc_o[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty + 16 * i;
            if (r < valid && o) {
                const size_t go = ((size_t)(t0 + r) * p.H + h) * D;
#pragma unroll
                for (int j = 0; j < NJ; ++j)
                    if (in_bounds(p.status, go + tx + 16 * j, n_tok))
                        o[go + tx + 16 * j] = from_f<Tin>(acc_o[i][j]);
            }
        }

        // ---- phase 6: S <- Diag(gamma) (S + Kb^T U)
        {
            constexpr int NI = D / 16;
            float acc[NI][NJ];
#pragma unroll
            for (int i = 0; i < NI; ++i)
#pragma unroll
                for (int j = 0; j < NJ; ++j) acc[i][j] = 0.f;
            for (int jr = 0; jr < C; ++jr) {
                float kb[NI], u[NJ];
#pragma unroll
                for (int i = 0; i < NI; ++i) kb[i] = sm.Kb[jr * LD + ty + 16 * i];
#pragma unroll
                for (int j = 0; j < NJ; ++j) u[j] = sm.Vb[jr * LD + tx + 16 * j];
#pragma unroll
                for (int i = 0; i < NI; ++i)
#pragma unroll
                    for (int j = 0; j < NJ; ++j) acc[i][j] = fmaf(kb[i], u[j], acc[i][j]);
            }
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int c = ty + 16 * i;
                const float g = sm.gam[c];
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    float &s = sm.S[c * LD + tx + 16 * j];
                    s = g * (s + acc[i][j]);
                }
            }
        }
    }
    __syncthreads();
    if (sref.S_T) {
        for (int idx = tid; idx < D * D; idx += kThreads) {
            const int vv = idx / D, c = idx % D;
            if (in_bounds(p.status, sref.off + idx, sref.ext))
                sref.S_T[sref.off + idx] = sm.S[c * LD + vv];
        }
    }
}

template <int D, typename Tin>
cudaError_t launch_typed(const FwdParams &p, cudaStream_t s) {
    const size_t smem = sizeof(SimtSmem<D>);
    auto kern = prefill_simt_kernel<D, Tin>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)((size_t)p.N * p.H), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const FwdParams &p, kda_dtype_t dt, cudaStream_t s) {
    if ((size_t)p.N * p.H == 0) return cudaSuccess;
    if (p.dk == 128)
        return dt == KDA_BF16 ? launch_typed<128, __nv_bfloat16>(p, s)
                              : launch_typed<128, float>(p, s);
    return dt == KDA_BF16 ? launch_typed<64, __nv_bfloat16>(p, s)
                          : launch_typed<64, float>(p, s);
}

}  // namespace kda

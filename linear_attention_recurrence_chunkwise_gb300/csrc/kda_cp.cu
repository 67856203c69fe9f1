// Segment-parallel (single-GPU context-parallel) forward.
//
// "Kimi K3模型架构详解" section 3.6 writes the effect of a sequence segment on
// the state as an affine map, S_out = M S_in + S~ (M: the segment's accumulated
// decay and erase acting on the incoming state; S~: the state the segment
// builds from zero), and composes such maps with (M2, b2) o (M1, b1) =
// (M2 M1, M2 b1 + b2).  Section 11.1 puts this on one GPU: when a rank holds
// few heads, most SMs idle during a long prefill, so the sequence is cut into
// segments that run side by side.
//
// Per sequence, P segments at chunk boundaries:
//   pass A  segment 0 from the real S0 (outputs and end state), and for every
//           later segment j two state-only runs: S~_j (from S0 = 0) and M_j
//           (v = 0 and S0 = I, so the end state is M_j I = M_j);
//   scan    S_in(1) = end of segment 0; S_in(j+1) = M_j S_in(j) + S~_j;
//   pass D  every later segment again from its S_in, writing its outputs; the
//           last one writes S_T.
// Both passes are the ordinary prefill kernels in task-table mode (one task per
// (range, initial state, final state, flags)), so they run on either engine.
// In memory the state is [v][c] = S^T, so the scan computes
// S_in(j+1)^T = S_in(j)^T M_j^T + S~_j^T, and the M run's memory image is M_j^T:
// a plain row-major product X M + S~ of the stored blocks.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kScanThreads = 256;

// Task tables, the zero V source, and the device check of cu_seqlens.
__global__ void __launch_bounds__(kPlanThreads) cp_plan_kernel(
    const int32_t *__restrict__ cu, int N, int T, int64_t Ttot, int P, int H, int d,
    const float *S0, float *S_T, CpLayout L, uint8_t *ws) {
    __shared__ int bad;
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    if (threadIdx.x == 0) {
        bad = 0;
        *status = KDA_OK;
    }
    uint4 *z = reinterpret_cast<uint4 *>(ws + L.vzero);
    for (size_t i = threadIdx.x; i < kVZeroBytes / 16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    if (cu) {
        for (int i = threadIdx.x; i <= N; i += blockDim.x) {
            const int32_t c = cu[i];
            const bool wrong = (i == 0 && c != 0) || (i == N && (int64_t)c != Ttot) ||
                               (i < N && cu[i + 1] < c);
            if (wrong) atomicExch(&bad, 1);
        }
        __syncthreads();
        if (bad) {
            if (threadIdx.x == 0) *status = KDA_ERR_INVALID_ARGUMENT;
            return;  // the prefill and scan kernels see the status and do nothing
        }
    }
    const size_t blk = (size_t)H * d * d;  // floats of one [H][d][d] state set
    SegTask *ta = reinterpret_cast<SegTask *>(ws + L.tasks_a);
    SegTask *td = reinterpret_cast<SegTask *>(ws + L.tasks_d);
    float *sa = reinterpret_cast<float *>(ws + L.s_a);
    float *st = reinterpret_cast<float *>(ws + L.s_t);
    float *mt = reinterpret_cast<float *>(ws + L.m_t);
    float *sin = reinterpret_cast<float *>(ws + L.s_in);
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        const int64_t start = cu ? (int64_t)cu[n] : (int64_t)n * T;
        const int len = cu ? cu[n + 1] - cu[n] : T;
        const int64_t nch = (len + kChunk - 1) / kChunk;
        for (int j = 0; j < P; ++j) {
            const int64_t t_lo = (int64_t)j * nch / P * kChunk;
            const int64_t t_hi = min((int64_t)(j + 1) * nch / P * kChunk, (int64_t)len);
            const int64_t s0 = start + t_lo;
            const int32_t sl = (int32_t)max((int64_t)0, t_hi - t_lo);
            if (j == 0) {
                ta[(size_t)n * (2 * P - 1)] = {s0, sl, 0, S0 ? S0 + n * blk : nullptr,
                                               sa + n * blk};
                continue;
            }
            const size_t r = (size_t)n * (P - 1) + (j - 1);
            ta[(size_t)n * (2 * P - 1) + 2 * j - 1] = {s0, sl, kTaskNoOutput, nullptr, st + r * blk};
            ta[(size_t)n * (2 * P - 1) + 2 * j] = {
                s0, sl, kTaskVZero | kTaskS0Identity | kTaskNoOutput, nullptr, mt + r * blk};
            td[r] = {s0, sl, 0, sin + r * blk,
                     j == P - 1 && S_T ? S_T + n * blk : nullptr};
        }
    }
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// S_in of every later segment: X <- X M + S~ in fp32.  Row v of X M is row v
// of X times M, so the rows are independent: a block takes kScanRows rows of
// one (sequence, head) through all its segments, 16 threads per row, each
// D / 16 consecutive columns.  M_{j+1} lands in shared memory (cp.async, two
// buffers) while step j computes, and the thread's S~ values are loaded before
// its product, so a step waits on no global load.
constexpr int kScanRows = 16;
template <int D>
__global__ void __launch_bounds__(kScanThreads) cp_scan_kernel(int N, int P, int H,
                                                                CpLayout L, uint8_t *ws) {
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    if (*status == KDA_ERR_INVALID_ARGUMENT) return;
    extern __shared__ __align__(16) float cp_smem[];
    float *Mbuf = cp_smem;           // two M_j [a][c] buffers
    float *X = Mbuf + 2 * D * D;     // this block's rows of X [r][a]
    constexpr int kBlocks = D / kScanRows, kCols = D / 16;
    const int nh = blockIdx.x / kBlocks, v0 = kScanRows * (blockIdx.x % kBlocks);
    const int n = nh / H, h = nh % H, tid = threadIdx.x;
    const int r = tid / 16, c0 = kCols * (tid % 16);
    const size_t blk = (size_t)H * D * D, hoff = (size_t)h * D * D + (size_t)v0 * D;
    const float *sa = reinterpret_cast<const float *>(ws + L.s_a) + n * blk + hoff;
    const float *st = reinterpret_cast<const float *>(ws + L.s_t);
    const float *mt = reinterpret_cast<const float *>(ws + L.m_t);
    float *sin = reinterpret_cast<float *>(ws + L.s_in);
    auto seg = [&](int j) { return ((size_t)n * (P - 1) + (j - 1)) * blk; };  // segment j's sets
    // extents for the bounds-checked build: the per-sequence set and the
    // per-later-segment sets; a block whose rows would leave them does nothing
    const size_t n_sets = (size_t)N * (P - 1) * blk;
    if (!in_bounds(status, n * blk + hoff + (size_t)kScanRows * D - 1, (size_t)N * blk) ||
        (P > 1 && !in_bounds(status, seg(P - 1) + hoff + (size_t)kScanRows * D - 1, n_sets)))
        return;
    // M_j into buffer (j - 1) % 2; every thread copies the same pieces each time
    auto stage_m = [&](int j) {
        const float *mj = mt + seg(j) + (size_t)h * D * D;
        float *dst = Mbuf + ((j - 1) & 1) * D * D;
        for (int i = tid; i < D * D / 4; i += kScanThreads) cp_async16(dst + 4 * i, mj + 4 * i);
        cp_async_commit();
    };
    for (int i = tid; i < kScanRows * D / 4; i += kScanThreads)
        reinterpret_cast<float4 *>(X)[i] = reinterpret_cast<const float4 *>(sa)[i];
    if (P > 2) stage_m(1);
    for (int j = 1; j < P; ++j) {
        __syncthreads();  // X complete; the last product has read its M buffer
        for (int i = tid; i < kScanRows * D / 4; i += kScanThreads)
            reinterpret_cast<float4 *>(sin + seg(j) + hoff)[i] = reinterpret_cast<const float4 *>(X)[i];
        if (j == P - 1) break;
        float add[kCols];  // this thread's S~_j entries
        const float *stj = st + seg(j) + hoff + (size_t)r * D + c0;
#pragma unroll
        for (int k = 0; k < kCols; k += 4) {
            const float4 x4 = *reinterpret_cast<const float4 *>(stj + k);
            add[k] = x4.x, add[k + 1] = x4.y, add[k + 2] = x4.z, add[k + 3] = x4.w;
        }
        cp_async_wait_all();
        __syncthreads();  // M_j in place
        if (j + 1 < P - 1) stage_m(j + 1);
        const float *M = Mbuf + ((j - 1) & 1) * D * D;
        float acc[kCols];
#pragma unroll
        for (int k = 0; k < kCols; ++k) acc[k] = add[k];
        for (int a = 0; a < D; ++a) {
            const float x = X[r * D + a];
#pragma unroll
            for (int k = 0; k < kCols; k += 4) {
                const float4 m = *reinterpret_cast<const float4 *>(&M[a * D + c0 + k]);
                acc[k] = fmaf(x, m.x, acc[k]);
                acc[k + 1] = fmaf(x, m.y, acc[k + 1]);
                acc[k + 2] = fmaf(x, m.z, acc[k + 2]);
                acc[k + 3] = fmaf(x, m.w, acc[k + 3]);
            }
        }
        __syncthreads();  // every product has read X
#pragma unroll
        for (int k = 0; k < kCols; ++k) X[r * D + c0 + k] = acc[k];
    }
    cp_async_wait_all();  // nothing in flight at exit
}

}  // namespace

CpLayout cp_layout(int N, int H, int d, int P) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t n = N > 0 ? (size_t)N : 1;
    const size_t blk = (size_t)H * d * d * sizeof(float);
    const size_t later = n * (size_t)(P > 1 ? P - 1 : 0);
    CpLayout L;
    size_t off = 256;  // status word
    L.tasks_a = off;
    off = up(off + n * (size_t)(2 * P - 1) * sizeof(SegTask));
    L.tasks_d = off;
    off = up(off + later * sizeof(SegTask));
    L.vzero = off;
    off = up(off + kVZeroBytes);
    L.s_a = off;
    off = up(off + n * blk);
    L.s_t = off;
    off = up(off + later * blk);
    L.m_t = off;
    off = up(off + later * blk);
    L.s_in = off;
    off = up(off + later * blk);
    L.total = off;
    return L;
}

cudaError_t launch_fwd_cp(const FwdParams &base, kda_dtype_t dt, bool use_tc, int P,
                          void *workspace, cudaStream_t s) {
    const int N = base.N, H = base.H, d = base.dk;
    const CpLayout L = cp_layout(N, H, d, P);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cp_plan_kernel<<<1, kPlanThreads, 0, s>>>(base.cu_seqlens, N, base.T, base.Ttot, P, H, d,
                                               base.S0, base.S_T, L, ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || N == 0) return e;
    auto run = [&](size_t table, int ntasks) {
        FwdParams p = base;
        p.tasks = reinterpret_cast<const SegTask *>(ws + table);
        p.N = ntasks;
        p.S0 = nullptr;
        p.S_T = nullptr;
        p.cu_seqlens = nullptr;
        p.order = nullptr;
        p.vzero = ws + L.vzero;
        return use_tc ? launch_prefill_tc(p, s) : launch_prefill_simt(p, dt, s);
    };
    if ((e = run(L.tasks_a, N * (2 * P - 1))) != cudaSuccess) return e;
    const size_t smem = (2 * (size_t)d * d + (size_t)kScanRows * d) * sizeof(float);
    const unsigned grid = (unsigned)((size_t)N * H * (d / kScanRows));
    if (d == 128) {
        e = cudaFuncSetAttribute(cp_scan_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        cp_scan_kernel<128><<<grid, kScanThreads, smem, s>>>(N, P, H, L, ws);
    } else {
        cp_scan_kernel<64><<<grid, kScanThreads, smem, s>>>(N, P, H, L, ws);  // 36 KB
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return run(L.tasks_d, N * (P - 1));
}

}  // namespace kda

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
//   scan    S_in(1) = end of segment 0; S_in(j+1) = M_j S_in(j) + S~_j (fp32
//           accuracy from three tf32 tensor-core products per tile);
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

// x rounded to the nearest tf32 value (ties away from zero), as its fp32 bit
// pattern, and the remainder: x = hi + lo
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
    lo = __float_as_uint(x - __uint_as_float(hi));
}

// d (16 x 8, fp32) += a (16 x 8) b (8 x 8) with tf32 operands (mma.sync m16n8k8)
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// S_in of every later segment: X <- X M + S~ in fp32.  Row v of X M is row v
// of X times M, so the rows are independent: a block takes kScanRows = 16 rows
// of one (sequence, head) through all its segments.  The product is an m = 16
// tensor-core tile: warp w owns output columns D / 8 w .. + D / 8 (one or two
// m16n8 tiles), takes the k = 8 slices of X (A) and M (B) from shared memory
// and splits each operand into a tf32 high part and the remainder, so that
// high x high + high x low + low x high gives the product to fp32 accuracy
// (the low x low term is below it).  The accumulators start from S~.  M_{j+1}
// lands in shared memory (cp.async, two buffers) while step j computes; X and
// M rows are padded (4 and 8 floats) so that the fragment loads of a warp hit
// 32 different banks.
constexpr int kScanRows = 16;
template <int D>
constexpr size_t scan_smem_bytes() {
    return (2 * (size_t)D * (D + 8) + (size_t)kScanRows * (D + 4)) * sizeof(float);
}
template <int D>
__global__ void __launch_bounds__(kScanThreads) cp_scan_kernel(int N, int P, int H,
                                                                CpLayout L, uint8_t *ws) {
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    if (*status == KDA_ERR_INVALID_ARGUMENT) return;
    extern __shared__ __align__(16) float cp_smem[];
    constexpr int kLdM = D + 8, kLdX = D + 4;
    constexpr int kTiles = D / 64;  // m16n8 output tiles per warp (8 warps)
    float *Mbuf = cp_smem;                 // two M_j [a][c] buffers, rows of kLdM
    float *X = Mbuf + 2 * D * kLdM;        // this block's rows of X [r][a], rows of kLdX
    constexpr int kBlocks = D / kScanRows;
    const int nh = blockIdx.x / kBlocks, v0 = kScanRows * (blockIdx.x % kBlocks);
    const int n = nh / H, h = nh % H, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, g = lane >> 2, t4 = lane & 3;
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
        float *dst = Mbuf + ((j - 1) & 1) * D * kLdM;
        for (int i = tid; i < D * D / 4; i += kScanThreads) {
            const int a = i / (D / 4), c = 4 * (i % (D / 4));
            cp_async16(dst + a * kLdM + c, mj + a * D + c);
        }
        cp_async_commit();
    };
    for (int i = tid; i < kScanRows * D / 4; i += kScanThreads) {
        const int r = i / (D / 4), c = 4 * (i % (D / 4));
        *reinterpret_cast<float4 *>(X + r * kLdX + c) =
            *reinterpret_cast<const float4 *>(sa + r * D + c);
    }
    if (P > 2) stage_m(1);
    for (int j = 1; j < P; ++j) {
        __syncthreads();  // X complete; the last product has read its M buffer
        for (int i = tid; i < kScanRows * D / 4; i += kScanThreads) {
            const int r = i / (D / 4), c = 4 * (i % (D / 4));
            *reinterpret_cast<float4 *>(sin + seg(j) + hoff + r * D + c) =
                *reinterpret_cast<const float4 *>(X + r * kLdX + c);
        }
        if (j == P - 1) break;
        // an empty segment's map is exactly (I, 0): X passes through unchanged
        // (bit for bit, which the tensor-core product would not give)
        const SegTask *td = reinterpret_cast<const SegTask *>(ws + L.tasks_d);
        const bool empty = td[(size_t)n * (P - 1) + (j - 1)].len == 0;
        // accumulators start from this warp's entries of S~_j: tile nt covers
        // columns c0 .. c0 + 7; lane (g, t4) holds rows g, g + 8, columns
        // c0 + 2 t4, + 1
        float acc[kTiles][3][4];
        const float *stj = st + seg(j) + hoff;
#pragma unroll
        for (int nt = 0; nt < kTiles; ++nt) {
            const int col = (D / 8) * warp + 8 * nt + 2 * t4;
            const float2 s0 = *reinterpret_cast<const float2 *>(stj + (size_t)g * D + col);
            const float2 s1 = *reinterpret_cast<const float2 *>(stj + (size_t)(g + 8) * D + col);
            acc[nt][2][0] = s0.x, acc[nt][2][1] = s0.y, acc[nt][2][2] = s1.x, acc[nt][2][3] = s1.y;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][0][e] = acc[nt][1][e] = 0.f;
        }
        cp_async_wait_all();
        __syncthreads();  // M_j in place
        if (j + 1 < P - 1) stage_m(j + 1);
        if (empty) continue;  // (the next step's first barrier follows)
        const float *M = Mbuf + ((j - 1) & 1) * D * kLdM;
#pragma unroll 4
        for (int k0 = 0; k0 < D; k0 += 8) {
            uint32_t ah[4], al[4];  // A = X[r][k0 + k]: (g, t4), (g + 8, t4), (g, t4 + 4), (g + 8, t4 + 4)
            split_tf32(X[g * kLdX + k0 + t4], ah[0], al[0]);
            split_tf32(X[(g + 8) * kLdX + k0 + t4], ah[1], al[1]);
            split_tf32(X[g * kLdX + k0 + t4 + 4], ah[2], al[2]);
            split_tf32(X[(g + 8) * kLdX + k0 + t4 + 4], ah[3], al[3]);
#pragma unroll
            for (int nt = 0; nt < kTiles; ++nt) {
                const int c = (D / 8) * warp + 8 * nt + g;  // B = M[k0 + k][c]: k = t4, t4 + 4
                uint32_t bh0, bl0, bh1, bl1;
                split_tf32(M[(k0 + t4) * kLdM + c], bh0, bl0);
                split_tf32(M[(k0 + t4 + 4) * kLdM + c], bh1, bl1);
                mma_tf32(acc[nt][0], al, bh0, bh1);
                mma_tf32(acc[nt][1], ah, bl0, bl1);
                mma_tf32(acc[nt][2], ah, bh0, bh1);
            }
        }
        __syncthreads();  // every product has read X
#pragma unroll
        for (int nt = 0; nt < kTiles; ++nt) {
            const int col = (D / 8) * warp + 8 * nt + 2 * t4;
            float r[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) r[e] = (acc[nt][0][e] + acc[nt][1][e]) + acc[nt][2][e];
            *reinterpret_cast<float2 *>(X + g * kLdX + col) = make_float2(r[0], r[1]);
            *reinterpret_cast<float2 *>(X + (g + 8) * kLdX + col) = make_float2(r[2], r[3]);
        }
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
        p.blocked = 0;  // task-table mode runs the plain tensor-core variant
        return use_tc ? launch_prefill_tensorcore(p, dt, s) : launch_prefill_simt(p, dt, s);
    };
    if ((e = run(L.tasks_a, N * (2 * P - 1))) != cudaSuccess) return e;
    const unsigned grid = (unsigned)((size_t)N * H * (d / kScanRows));
    if (d == 128) {
        constexpr size_t smem = scan_smem_bytes<128>();  // 146 KB
        e = cudaFuncSetAttribute(cp_scan_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        cp_scan_kernel<128><<<grid, kScanThreads, smem, s>>>(N, P, H, L, ws);
    } else {
        constexpr size_t smem = scan_smem_bytes<64>();  // 40 KB
        e = cudaFuncSetAttribute(cp_scan_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        cp_scan_kernel<64><<<grid, kScanThreads, smem, s>>>(N, P, H, L, ws);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return run(L.tasks_d, N * (P - 1));
}

}  // namespace kda

// Host side of the libkda C ABI: argument validation, engine choice and
// launches.  Nothing here allocates, frees or synchronises (except
// kda_read_device_status, whose job is to read a device word).
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kda_internal.h"

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned(const void *p, unsigned bytes) { return ((uintptr_t)p & (bytes - 1)) == 0; }

bool fault_injected() {
    // Host-only failure injection for tests of the error path: with
    // KDA_FAULT_INJECT=launch the entry points report a launch failure
    // without enqueueing anything.
    const char *e = getenv("KDA_FAULT_INJECT");
    return e && strcmp(e, "launch") == 0;
}

bool supported_dims(int dk, int dv) { return dk == dv && (dk == 64 || dk == 128); }

}  // namespace

extern "C" {

size_t kda_fwd_workspace_bytes(int N) {
    const size_t n = N > 0 ? (size_t)N : 1;
    return (kda::kWsOrderOffset + 4 * n + 15) & ~(size_t)15;
}

const char *kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_DOMAIN: return "KDA_ERR_DOMAIN";
        case KDA_ERR_BOUNDS: return "KDA_ERR_BOUNDS";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    }
    return "KDA_ERR_UNKNOWN";
}

size_t kda_state_bytes(int layers, int N, int H, int d_k, int d_v, int elem_bytes) {
    const int f[6] = {layers, N, H, d_k, d_v, elem_bytes};
    size_t total = 1;
    for (int i = 0; i < 6; ++i) {
        if (f[i] < 0) return 0;
        if (f[i] != 0 && total > SIZE_MAX / (size_t)f[i]) return 0;
        total *= (size_t)f[i];
    }
    return total;
}

}  // extern "C"

namespace {

// Argument checks shared by kda_fwd and kda_fwd_cp (everything but the
// workspace size), and the engine choice.  On KDA_OK, p holds the arguments.
kda_status_t check_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                       const float *beta, const float *S0, const int32_t *cu_seqlens, int B,
                       int T, int H, int d_k, int d_v, int N, kda_dtype_t dtype, void *o,
                       float *S_T, void *workspace, kda_engine_t engine, kda::FwdParams &p,
                       bool &use_tc) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (engine != KDA_ENGINE_AUTO && engine != KDA_ENGINE_TENSORCORE &&
        engine != KDA_ENGINE_CUDACORE && engine != KDA_ENGINE_TENSORCORE_WIDE)
        return KDA_ERR_INVALID_ARGUMENT;
    if (B < 0 || T < 0 || N < 0 || H <= 0 || d_k <= 0 || d_v <= 0)
        return KDA_ERR_INVALID_ARGUMENT;
    if (!supported_dims(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if (cu_seqlens) {
        if (B != 1) return KDA_ERR_INVALID_ARGUMENT;
        if (((uintptr_t)cu_seqlens & 3u) != 0) return KDA_ERR_INVALID_ARGUMENT;
    } else if (N != B) {
        return KDA_ERR_INVALID_ARGUMENT;
    }
    const int64_t Ttot = (int64_t)B * T;
    if ((int64_t)N * H > INT32_MAX) return KDA_ERR_INVALID_ARGUMENT;
    if (Ttot > 0) {
        if (!q || !k || !v || !log_alpha || !beta || !o) return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
            !aligned(beta, 4) || !aligned16(o))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    if ((S0 && !aligned16(S0)) || (S_T && !aligned16(S_T))) return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace) return KDA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KDA_ERR_INVALID_ARGUMENT;

    // tensor cores: bf16 at d = 128 (the blocked path for wide gates only there),
    // fp32 or bf16 at d = 64
    const bool tc_ok = kda::prefill_tc_supported(dtype, d_k, d_v) && Ttot <= INT32_MAX;
    const bool tc64_ok = d_k == 64 && d_v == 64 && Ttot <= INT32_MAX;
    if (engine == KDA_ENGINE_TENSORCORE_WIDE && !tc_ok) return KDA_ERR_UNSUPPORTED;
    if (engine == KDA_ENGINE_TENSORCORE && !(tc_ok || tc64_ok)) return KDA_ERR_UNSUPPORTED;
    // AUTO: the tensor cores wherever they run (at d = 64 they take 0.6 of the
    // CUDA-core engine's time for fp32 inputs and 0.55 for bf16, measured)
    use_tc = engine == KDA_ENGINE_TENSORCORE || engine == KDA_ENGINE_TENSORCORE_WIDE ||
             (engine == KDA_ENGINE_AUTO && (tc_ok || tc64_ok));

    p = kda::FwdParams{};
    p.tasks = nullptr;
    p.vzero = nullptr;
    p.q = q;
    p.k = k;
    p.v = v;
    p.log_alpha = log_alpha;
    p.beta = beta;
    p.S0 = S0;
    p.cu_seqlens = cu_seqlens;
    p.o = o;
    p.S_T = S_T;
    p.status = static_cast<int32_t *>(workspace);
    p.order = cu_seqlens ? reinterpret_cast<const int32_t *>(
                               static_cast<char *>(workspace) + kda::kWsOrderOffset)
                         : nullptr;
    p.Ttot = Ttot;
    p.T = T;
    p.H = H;
    p.N = N;
    p.dk = d_k;
    p.dv = d_v;
    p.blocked = engine == KDA_ENGINE_TENSORCORE_WIDE;
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_fwd_engine(const void *q, const void *k, const void *v,
                            const float *log_alpha, const float *beta, const float *S0,
                            const int32_t *cu_seqlens, int B, int T, int H, int d_k,
                            int d_v, int N, kda_dtype_t dtype, void *o, float *S_T,
                            void *workspace, size_t workspace_bytes, void *stream,
                            kda_engine_t engine) {
    kda::FwdParams p;
    bool use_tc = false;
    const kda_status_t st = check_fwd(q, k, v, log_alpha, beta, S0, cu_seqlens, B, T, H, d_k,
                                      d_v, N, dtype, o, S_T, workspace, engine, p, use_tc);
    if (st != KDA_OK) return st;
    if (workspace_bytes < kda_fwd_workspace_bytes(N)) return KDA_ERR_WORKSPACE;
    if (fault_injected()) return KDA_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kda::launch_schedule(p, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (N == 0) return KDA_OK;
    const cudaError_t e = use_tc ? kda::launch_prefill_tensorcore(p, dtype, s)
                                 : kda::launch_prefill_simt(p, dtype, s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_gated_rmsnorm(const void *o, const void *g, const float *norm_weight,
                               float eps, int64_t rows, int d_v, kda_dtype_t dtype, void *y,
                               void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (rows < 0 || d_v <= 0 || !(eps >= 0.f) || eps > 3.0e38f) return KDA_ERR_INVALID_ARGUMENT;
    if (d_v != 64 && d_v != 128) return KDA_ERR_UNSUPPORTED;
    if (rows == 0) return KDA_OK;
    if (!o || !g || !y || !aligned16(o) || !aligned16(g) || !aligned16(y) ||
        (norm_weight && !aligned(norm_weight, 4)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (fault_injected()) return KDA_ERR_CUDA;
    const cudaError_t e = kda::launch_gated_rmsnorm(o, g, norm_weight, eps, rows, d_v, dtype, y,
                                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_short_conv(const void *xq, const void *xk, const void *xv, const float *wq,
                            const float *wk, const float *wv, const float *conv0,
                            const int32_t *cu_seqlens, int B, int T, int H, int d, int N,
                            kda_dtype_t dtype, float eps, void *q, void *k, void *v,
                            float *conv_T, void *workspace, size_t workspace_bytes,
                            void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (B < 0 || T < 0 || N < 0 || H <= 0 || d <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!(eps >= 0.f) || eps > 3.0e38f) return KDA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return KDA_ERR_UNSUPPORTED;
    if (cu_seqlens) {
        if (B != 1 || ((uintptr_t)cu_seqlens & 3u) != 0) return KDA_ERR_INVALID_ARGUMENT;
    } else if (N != B) {
        return KDA_ERR_INVALID_ARGUMENT;
    }
    const int64_t Ttot = (int64_t)B * T;
    if ((int64_t)N * H > INT32_MAX / 9) return KDA_ERR_INVALID_ARGUMENT;
    const void *x[3] = {xq, xk, xv};
    const float *w[3] = {wq, wk, wv};
    void *y[3] = {q, k, v};
    for (int i = 0; i < 3; ++i) {
        if (Ttot > 0 && (!x[i] || !y[i] || !aligned16(x[i]) || !aligned16(y[i])))
            return KDA_ERR_INVALID_ARGUMENT;
        if (!w[i] || !aligned16(w[i])) return KDA_ERR_INVALID_ARGUMENT;
    }
    if ((conv0 && !aligned16(conv0)) || (conv_T && !aligned16(conv_T)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace) return KDA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KDA_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < kda_fwd_workspace_bytes(N)) return KDA_ERR_WORKSPACE;
    if (fault_injected()) return KDA_ERR_CUDA;
    // the status word and the device-side check of cu_seqlens, as in kda_fwd
    kda::FwdParams p{};
    p.cu_seqlens = cu_seqlens;
    p.N = N;
    p.Ttot = Ttot;
    p.status = static_cast<int32_t *>(workspace);
    p.order = cu_seqlens ? reinterpret_cast<const int32_t *>(
                               static_cast<char *>(workspace) + kda::kWsOrderOffset)
                         : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kda::launch_schedule(p, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (N == 0) return KDA_OK;
    const cudaError_t e = kda::launch_short_conv(x, w, conv0, cu_seqlens, Ttot, T, H, d, N, dtype,
                                                 eps, y, conv_T, p.status, false, s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_short_conv_step(const void *xq, const void *xk, const void *xv,
                                 const float *wq, const float *wk, const float *wv, float *conv,
                                 int N, int H, int d, kda_dtype_t dtype, float eps, void *q,
                                 void *k, void *v, void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || H <= 0 || d <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!(eps >= 0.f) || eps > 3.0e38f) return KDA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)N * H > INT32_MAX / 9) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    const void *x[3] = {xq, xk, xv};
    const float *w[3] = {wq, wk, wv};
    void *y[3] = {q, k, v};
    for (int i = 0; i < 3; ++i)
        if (!x[i] || !y[i] || !w[i] || !aligned16(x[i]) || !aligned16(y[i]) || !aligned16(w[i]))
            return KDA_ERR_INVALID_ARGUMENT;
    if (!conv || !aligned16(conv)) return KDA_ERR_INVALID_ARGUMENT;
    if (fault_injected()) return KDA_ERR_CUDA;
    const cudaError_t e = kda::launch_short_conv(x, w, nullptr, nullptr, N, 1, H, d, N, dtype, eps,
                                                 y, conv, nullptr, true,
                                                 static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_layer_step(const void *xq, const void *xk, const void *xv,
                                   const float *wq, const float *wk, const float *wv, float *conv,
                                   float l2_eps, const float *log_alpha, const float *beta,
                                   float *S, int N, int H, int d, kda_dtype_t dtype,
                                   const void *g, const float *norm_weight, float eps, void *y,
                                   void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || H <= 0 || d <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!(eps >= 0.f) || eps > 3.0e38f || !(l2_eps >= 0.f) || l2_eps > 3.0e38f)
        return KDA_ERR_INVALID_ARGUMENT;
    if (d != 64 && d != 128) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)N * H > INT32_MAX / 9) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    const void *x[3] = {xq, xk, xv};
    const float *w[3] = {wq, wk, wv};
    for (int i = 0; i < 3; ++i)
        if (!x[i] || !w[i] || !aligned16(x[i]) || !aligned16(w[i])) return KDA_ERR_INVALID_ARGUMENT;
    if (!conv || !log_alpha || !beta || !S || !g || !y || !aligned16(conv) ||
        !aligned16(log_alpha) || !aligned(beta, 4) || !aligned16(S) || !aligned16(g) ||
        !aligned16(y) || (norm_weight && !aligned(norm_weight, 4)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (fault_injected()) return KDA_ERR_CUDA;
    const cudaError_t e = kda::launch_decode_layer(x, w, conv, l2_eps, log_alpha, beta, S, N, H, d,
                                                   dtype, g, norm_weight, eps, y,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_fwd_gated(const void *q, const void *k, const void *v, const float *log_alpha,
                           const float *beta, const float *S0, const int32_t *cu_seqlens,
                           int B, int T, int H, int d_k, int d_v, int N, kda_dtype_t dtype,
                           const void *g, const float *norm_weight, float eps, void *y,
                           float *S_T, void *workspace, size_t workspace_bytes, void *stream,
                           kda_engine_t engine, kda_epilogue_t mode) {
    if (mode != KDA_EPILOGUE_AUTO && mode != KDA_EPILOGUE_FUSED && mode != KDA_EPILOGUE_SEPARATE)
        return KDA_ERR_INVALID_ARGUMENT;
    kda::FwdParams p;
    bool use_tc = false;
    const kda_status_t st = check_fwd(q, k, v, log_alpha, beta, S0, cu_seqlens, B, T, H, d_k,
                                      d_v, N, dtype, y, S_T, workspace, engine, p, use_tc);
    if (st != KDA_OK) return st;
    if (!(eps >= 0.f) || eps > 3.0e38f) return KDA_ERR_INVALID_ARGUMENT;
    if (p.Ttot > 0 && (!g || !aligned16(g))) return KDA_ERR_INVALID_ARGUMENT;
    if (norm_weight && !aligned(norm_weight, 4)) return KDA_ERR_INVALID_ARGUMENT;
    if (mode == KDA_EPILOGUE_FUSED && (!use_tc || p.blocked || d_k != 128)) return KDA_ERR_UNSUPPORTED;
    if (workspace_bytes < kda_fwd_workspace_bytes(N)) return KDA_ERR_WORKSPACE;
    if (fault_injected()) return KDA_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (kda::launch_schedule(p, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (N == 0) return KDA_OK;
    cudaError_t e;
    if (mode == KDA_EPILOGUE_FUSED) {  // in the tensor-core kernel's output stores
        p.gate = g;
        p.norm_w = norm_weight;
        p.eps = eps;
        e = kda::launch_prefill_tc(p, s);
    } else {  // o into y, then the epilogue in place (measured faster: AUTO)
        e = use_tc ? kda::launch_prefill_tensorcore(p, dtype, s) : kda::launch_prefill_simt(p, dtype, s);
        if (e == cudaSuccess)
            e = kda::launch_gated_rmsnorm(y, g, norm_weight, eps, p.Ttot * H, d_v, dtype, y, s);
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

size_t kda_fwd_cp_workspace_bytes(int N, int H, int d_k, int d_v, int segments) {
    if (segments < 1 || H <= 0 || !supported_dims(d_k, d_v)) return 0;
    const size_t base = kda_fwd_workspace_bytes(N);
    if (segments == 1) return base;
    const size_t cp = kda::cp_layout(N, H, d_k, segments).total;
    return cp > base ? cp : base;
}

int kda_fwd_cp_segments(int N, int H, int64_t Ttot) {
    if (N <= 0 || H <= 0 || Ttot <= 0) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return 1;
    // Modelled time in chunk periods of one block (one block per SM): a plain
    // pass walks every chunk of a sequence in ceil(N H / SMs) waves; P >= 2
    // segments walk a segment in pass A (N H (2P - 1) blocks) and again in
    // pass D (N H (P - 1) blocks), plus P - 2 scan steps of about 2.5 periods
    // (measured on the long prefill) and a few periods of launch and pipeline
    // fill.
    const int64_t units = (int64_t)N * H;
    const int64_t chunks = (Ttot / N + 63) / 64;  // per sequence, on average
    auto waves = [&](int64_t blocks) { return (double)((blocks + sms - 1) / sms); };
    int best = 1;
    double best_t = waves(units) * (double)chunks;
    for (int64_t P = 2; P <= chunks && P <= 1024; ++P) {
        const double seg = (double)((chunks + P - 1) / P);
        const double t = (waves(units * (2 * P - 1)) + waves(units * (P - 1))) * seg +
                         2.5 * (double)(P - 2) + 6.0;
        if (t < best_t) {
            best_t = t;
            best = (int)P;
        }
    }
    return best;
}

kda_status_t kda_fwd_cp(const void *q, const void *k, const void *v, const float *log_alpha,
                        const float *beta, const float *S0, const int32_t *cu_seqlens, int B,
                        int T, int H, int d_k, int d_v, int N, kda_dtype_t dtype, void *o,
                        float *S_T, int segments, void *workspace, size_t workspace_bytes,
                        void *stream, kda_engine_t engine) {
    kda::FwdParams p;
    bool use_tc = false;
    const kda_status_t st = check_fwd(q, k, v, log_alpha, beta, S0, cu_seqlens, B, T, H, d_k,
                                      d_v, N, dtype, o, S_T, workspace, engine, p, use_tc);
    if (st != KDA_OK) return st;
    if (segments < 1 || segments > 65536) return KDA_ERR_INVALID_ARGUMENT;
    if ((int64_t)N * H * (2 * (int64_t)segments - 1) > INT32_MAX) return KDA_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < kda_fwd_cp_workspace_bytes(N, H, d_k, d_v, segments))
        return KDA_ERR_WORKSPACE;
    if (segments == 1)
        return kda_fwd_engine(q, k, v, log_alpha, beta, S0, cu_seqlens, B, T, H, d_k, d_v, N,
                              dtype, o, S_T, workspace, workspace_bytes, stream, engine);
    if (fault_injected()) return KDA_ERR_CUDA;
    const cudaError_t e = kda::launch_fwd_cp(p, dtype, use_tc, segments, workspace,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                     const float *beta, const float *S0, const int32_t *cu_seqlens, int B,
                     int T, int H, int d_k, int d_v, int N, kda_dtype_t dtype, void *o,
                     float *S_T, void *workspace, size_t workspace_bytes, void *stream) {
    return kda_fwd_engine(q, k, v, log_alpha, beta, S0, cu_seqlens, B, T, H, d_k, d_v, N,
                          dtype, o, S_T, workspace, workspace_bytes, stream,
                          KDA_ENGINE_AUTO);
}

kda_status_t kda_decode_step(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta, float *S, int N,
                             int H, int d_k, int d_v, kda_dtype_t dtype, void *o,
                             void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || H <= 0 || d_k <= 0 || d_v <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!supported_dims(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)N * H > INT32_MAX) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !S || !o) return KDA_ERR_INVALID_ARGUMENT;
    const unsigned elem = dtype == KDA_BF16 ? 2u : 4u;
    if (!aligned(q, elem) || !aligned(k, elem) || !aligned(v, elem) || !aligned(o, elem) ||
        !aligned(log_alpha, 4) || !aligned(beta, 4) || !aligned16(S))
        return KDA_ERR_INVALID_ARGUMENT;
    if (fault_injected()) return KDA_ERR_CUDA;
    const cudaError_t e = kda::launch_decode(q, k, v, log_alpha, beta, S, N, H, d_k, dtype, o,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_step_gated(const void *q, const void *k, const void *v,
                                   const float *log_alpha, const float *beta, float *S, int N,
                                   int H, int d_k, int d_v, kda_dtype_t dtype, const void *g,
                                   const float *norm_weight, float eps, void *y, void *stream,
                                   kda_epilogue_t mode) {
    if (mode != KDA_EPILOGUE_AUTO && mode != KDA_EPILOGUE_FUSED && mode != KDA_EPILOGUE_SEPARATE)
        return KDA_ERR_INVALID_ARGUMENT;
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || H <= 0 || d_k <= 0 || d_v <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!(eps >= 0.f) || eps > 3.0e38f) return KDA_ERR_INVALID_ARGUMENT;
    if (!supported_dims(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)N * H > INT32_MAX) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !S || !y || !g) return KDA_ERR_INVALID_ARGUMENT;
    const unsigned elem = dtype == KDA_BF16 ? 2u : 4u;
    if (!aligned(q, elem) || !aligned(k, elem) || !aligned(v, elem) || !aligned(y, elem) ||
        !aligned(g, elem) || !aligned(log_alpha, 4) || !aligned(beta, 4) || !aligned16(S) ||
        (norm_weight && !aligned(norm_weight, 4)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (fault_injected()) return KDA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (mode == KDA_EPILOGUE_SEPARATE) {
        e = kda::launch_decode(q, k, v, log_alpha, beta, S, N, H, d_k, dtype, y, s);
        if (e == cudaSuccess)
            e = kda::launch_gated_rmsnorm(y, g, norm_weight, eps, (int64_t)N * H, d_v, dtype, y, s);
    } else {  // fused (measured faster: AUTO)
        e = kda::launch_decode(q, k, v, log_alpha, beta, S, N, H, d_k, dtype, y, s, g,
                               norm_weight, eps);
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

static kda_status_t check_draft_args(const void *q, const void *k, const void *v,
                                     const float *log_alpha, const float *beta, const float *S,
                                     int N, int K, int H, int d_k, int d_v, kda_dtype_t dtype) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || H <= 0 || d_k <= 0 || d_v <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (K < 1 || K > KDA_MAX_DRAFT_TOKENS) return KDA_ERR_INVALID_ARGUMENT;
    if (!supported_dims(d_k, d_v)) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)N * K * H > INT32_MAX) return KDA_ERR_INVALID_ARGUMENT;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !S) return KDA_ERR_INVALID_ARGUMENT;
    const unsigned elem = dtype == KDA_BF16 ? 2u : 4u;
    if (!aligned(q, elem) || !aligned(k, elem) || !aligned(v, elem) || !aligned(log_alpha, 4) ||
        !aligned(beta, 4) || !aligned16(S))
        return KDA_ERR_INVALID_ARGUMENT;
    return KDA_OK;
}

kda_status_t kda_verify_tokens(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, const float *S,
                               int N, int K, int H, int d_k, int d_v, kda_dtype_t dtype,
                               void *o, void *stream) {
    const kda_status_t st = check_draft_args(q, k, v, log_alpha, beta, S, N, K, H, d_k, d_v,
                                             dtype);
    if (st != KDA_OK || N == 0) return st;
    if (!o || !aligned(o, dtype == KDA_BF16 ? 2u : 4u)) return KDA_ERR_INVALID_ARGUMENT;
    if (fault_injected()) return KDA_ERR_CUDA;
    const cudaError_t e = kda::launch_verify(q, k, v, log_alpha, beta, S, N, K, H, d_k, dtype,
                                             o, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_commit_tokens(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, float *S,
                               const int32_t *n_accept, int N, int K, int H, int d_k, int d_v,
                               kda_dtype_t dtype, void *stream) {
    const kda_status_t st = check_draft_args(q, k, v, log_alpha, beta, S, N, K, H, d_k, d_v,
                                             dtype);
    if (st != KDA_OK || N == 0) return st;
    if (n_accept && !aligned(n_accept, 4)) return KDA_ERR_INVALID_ARGUMENT;
    if (fault_injected()) return KDA_ERR_CUDA;
    const cudaError_t e = kda::launch_commit(q, k, v, log_alpha, beta, S, n_accept, N, K, H,
                                             d_k, dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_read_device_status(const void *workspace, size_t workspace_bytes,
                                    void *stream) {
    if (!workspace || workspace_bytes < 4) return KDA_ERR_WORKSPACE;
    int32_t word = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    return static_cast<kda_status_t>(word);
}

}  // extern "C"

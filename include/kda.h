/*
 * kda.h -- C ABI of libkda, a single-GPU (sm_103a) implementation of the
 * Kimi Delta Attention (KDA) operator.
 *
 * The operator, per sequence and head, with state S in R^{d_k x d_v}:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t                       (the read sees the token's own write)
 *
 * defined in "Kimi K3 的 KDA：1M context 不必把所有 KV 都留下" section 3,
 * "Kimi K3模型架构详解" section 3.2 and "Kimi Delta Attention 完全拆解" (the KDA
 * equations with the decayed state Diag(alpha) S and the per-token decode order).
 * alpha_t = exp(log_alpha_t) is a per-key-channel gate; the library takes the
 * gate in the log domain, as the pages' implementations do ("完全拆解": g holds
 * log alpha and is accumulated with a cumulative sum before exponentiation).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is caller-owned DEVICE memory (cudaMalloc, a caching
 *    allocator, ...), contiguous and row-major.  kda_fwd needs q, k, v,
 *    log_alpha, o, S0, S_T and the workspace 16-byte aligned; beta and
 *    cu_seqlens need their natural (4-byte) alignment.  kda_decode_step needs
 *    S 16-byte aligned and the per-token vectors naturally aligned.  The library
 *    never allocates, frees or synchronises, except kda_read_device_status,
 *    which synchronises the given stream to read the status word.
 *  - `stream` is a cudaStream_t passed as void*; NULL selects the legacy
 *    default stream.  All work is enqueued asynchronously on it.  kda_fwd,
 *    kda_fwd_engine, kda_fwd_cp and kda_decode_step only enqueue kernels, so
 *    a stream capture records them into a CUDA graph whose replays give the
 *    same results as eager calls (make one eager call first: it performs the
 *    one-time host set-up).
 *  - The state is fp32 and laid out [N, H, d_v, d_k] (key channel innermost):
 *    memory element [n][h][v][c] holds the logical S[c][v].  This is the
 *    [batch, heads, value_dim, key_dim] layout "Kimi K3 混合线性注意力" section 3
 *    reports for FlashKDA.
 *  - log_alpha and beta are fp32.  q, k, v and o are all of one dtype
 *    (kda_dtype_t).  q and k are used as given; the pages put the L2
 *    normalisation of q and k in the parameterisation before the operator
 *    ("完全拆解", KDA layer parameterisation), so the caller applies it.
 *  - Preconditions: log_alpha finite and <= 0 (alpha in (0, 1]); beta finite.
 *  - Argument errors are reported by the return code before anything is
 *    enqueued.  A failed kernel launch returns KDA_ERR_CUDA.  Conditions only
 *    the GPU can see (see kda_fwd) set a status word in the workspace, read
 *    with kda_read_device_status; the kernels never trap.
 *  - Supported: d_k = d_v in {64, 128}.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size, bad dtype */
    KDA_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. d_k != d_v) */
    KDA_ERR_WORKSPACE = 3,        /* workspace missing or smaller than required */
    KDA_ERR_CUDA = 4,             /* a CUDA call or kernel launch failed */
    KDA_ERR_DOMAIN = 5,           /* reserved: no entry point of this version raises it
                                     (every finite gate is supported) */
    KDA_ERR_TIMEOUT = 6,          /* device status: a kernel wait gave up (not expected) */
    KDA_ERR_BOUNDS = 7            /* device status, bounds-checked build only: an index
                                     outside its tensor was found and the access skipped */
} kda_status_t;

typedef enum {
    KDA_F32 = 0,  /* q, k, v, o are float */
    KDA_BF16 = 1  /* q, k, v, o are bfloat16 (round-to-nearest-even output) */
} kda_dtype_t;

typedef enum {
    KDA_ENGINE_AUTO = 0,        /* the tensor-core engine where it runs (bf16 at d = 128,
                                   any dtype at d = 64), else the CUDA-core engine */
    KDA_ENGINE_TENSORCORE = 1,  /* tcgen05 kernels: bf16 at d = 128 (TMA, warp-specialised);
                                   fp32 or bf16 at d = 64, to fp32 accuracy (every operand a
                                   bf16 hi/lo pair, three products per K slice) */
    KDA_ENGINE_CUDACORE = 2,    /* fp32 CUDA-core chunkwise kernel: any supported dtype/d */
    KDA_ENGINE_TENSORCORE_WIDE = 3  /* the tensor-core kernel with the blocked path for
                                       chunks outside the chunk form's log-decay range
                                       (see kda_fwd, gate domain): for gates like K3's
                                       (per-token log-decay down to -5); a few percent
                                       slower than KDA_ENGINE_TENSORCORE on gates that
                                       stay in range.  Plain kda_fwd / kda_fwd_engine /
                                       kda_fwd_gated calls (separate epilogue) only;
                                       kda_fwd_cp treats it as KDA_ENGINE_TENSORCORE */
} kda_engine_t;

/* Bytes of workspace kda_fwd needs for N sequences (status word and the
 * longest-first launch order).  Never zero; independent of T. */
size_t kda_fwd_workspace_bytes(int N);

/*
 * kda_fwd -- chunkwise-parallel forward (prefill) over whole sequences.
 *
 * Computes o_t for every token and the final state S_T of every (sequence,
 * head), starting from S0.  Execution form: 64-token chunks; within a chunk the
 * cumulative log-decay, the WY/UT-style lower-triangular solve and the
 * intra-chunk masked contractions run in parallel; between chunks the state
 * is handed on, S <- Diag(gamma_C) S + (Gamma^{i->C} . K)^T (U - W S)
 * ("完全拆解", chunkwise parallelism and the hardware-aware kernel;
 * "Kimi K3 的 KDA" section 5; "Kimi K3模型架构详解" section 3.5).
 *
 * Layout (Ttot = B*T tokens, or the packed total with cu_seqlens):
 *   q, k       [Ttot, H, d_k]   dtype          v, o  [Ttot, H, d_v]  dtype
 *   log_alpha  [Ttot, H, d_k]   fp32           beta  [Ttot, H]       fp32
 *   S0         [N, H, d_v, d_k] fp32, or NULL for a zero initial state
 *   S_T        [N, H, d_v, d_k] fp32, or NULL to skip; may alias S0 exactly
 *   cu_seqlens [N+1] int32 device offsets (cu_seqlens[0] = 0, non-decreasing,
 *              cu_seqlens[N] = Ttot), or NULL for a fixed-length batch, in which
 *              case N must equal B and sequence b owns tokens b*T .. b*T+T-1.
 *   With cu_seqlens, pass B = 1 and T = Ttot.  Zero-length sequences are
 *   allowed (S_T = S0).  Sequences never interact.
 *   workspace  device memory of at least kda_fwd_workspace_bytes(N) bytes,
 *              16-byte aligned; its contents on entry do not matter.
 *
 * Gate domain: any finite log_alpha <= 0.  The chunk form scales keys by
 * exp(-G), G the in-chunk cumulative log-decay, which overflows fp32 once |G|
 * passes 80 -- reachable under K3's per-token bound of -5 ("Kimi K3 的 KDA"
 * section 6: -320 over 64 tokens).  KDA_ENGINE_TENSORCORE_WIDE keeps such a
 * chunk on the tensor cores when each of its four 16-token blocks stays within
 * 80 (always, under K3's bound): A and M are built block by block with the
 * decay referenced to each block's first token ("Kimi K3模型架构详解" section
 * 3.4), and the state is handed on as Diag(gamma) S + K~^T U with K~ the keys
 * decayed to the chunk end.  Any other such chunk is computed token by token
 * with the recurrence itself on CUDA cores, in fp32: by the CUDA-core engine
 * chunk by chunk, by the tensor-core engines for the whole (sequence, head)
 * that contains one (from S0, after its chunk pass; S_T may still alias S0).
 *
 * Device status (kda_read_device_status): KDA_ERR_INVALID_ARGUMENT when the
 * device-side cu_seqlens is not non-decreasing or does not end at Ttot; no
 * output is written then.  KDA_ERR_TIMEOUT if a wait inside the tensor-core
 * kernel exceeded its time limit (outputs undefined; the kernel still exits
 * and releases its resources).
 */
kda_status_t kda_fwd(const void *q, const void *k, const void *v,
                     const float *log_alpha, const float *beta, const float *S0,
                     const int32_t *cu_seqlens, int B, int T, int H, int d_k, int d_v,
                     int N, kda_dtype_t dtype, void *o, float *S_T,
                     void *workspace, size_t workspace_bytes, void *stream);

/* kda_fwd with an explicit engine choice (for tests and benchmarks).
 * KDA_ERR_UNSUPPORTED if the engine cannot run this dtype/size. */
kda_status_t kda_fwd_engine(const void *q, const void *k, const void *v,
                            const float *log_alpha, const float *beta, const float *S0,
                            const int32_t *cu_seqlens, int B, int T, int H, int d_k,
                            int d_v, int N, kda_dtype_t dtype, void *o, float *S_T,
                            void *workspace, size_t workspace_bytes, void *stream,
                            kda_engine_t engine);

/*
 * kda_fwd_cp -- segment-parallel ("context-parallel" on one GPU) forward.
 *
 * Same arguments, results and conventions as kda_fwd_engine, for prefills that
 * leave SMs idle: one (sequence, head) is one serial chain of chunks, so with
 * few heads -- a rank that holds a tensor-parallel share of the heads -- most
 * of the GPU waits ("Kimi K3模型架构详解" section 11.1: single-GPU SM-level
 * context parallelism over sequence segments).  Each sequence is cut into
 * `segments` pieces at 64-token chunk boundaries.  A segment acts on the state
 * as the affine map S_out = M S_in + S~ (section 3.6: M the segment's
 * accumulated decay and erase, S~ the state it builds from zero; maps compose
 * as (M2, b2) o (M1, b1) = (M2 M1, M2 b1 + b2)).  The call runs, on `stream`:
 * the first segment of every sequence from S0 together with (S~, M) of every
 * later segment (M as the end state from S0 = I with v = 0); an fp32 scan that
 * composes the maps into each later segment's start state; then the later
 * segments again from their start states, which writes their outputs and S_T.
 * The later segments thus cost about three times a plain pass, in parallel.
 *
 * segments: >= 1 (1 is kda_fwd_engine); kda_fwd_cp_segments suggests a value.
 *   Sequences shorter than `segments` chunks get empty segments (identity
 *   maps).  Requires d_k = d_v (as every entry point here).
 * workspace: at least kda_fwd_cp_workspace_bytes(N, H, d_k, d_v, segments)
 *   bytes, 16-byte aligned, contents on entry irrelevant; it holds the status
 *   word (kda_read_device_status), the segment task tables and four fp32
 *   state sets per later segment: about 4 (segments - 1) N H d_k d_v 4 bytes.
 * S_T may alias S0.  Results agree with kda_fwd to the rounding of the state
 * hand-off: the maps of the tensor-core engine carry its bf16 operand
 * rounding, which the scan composes; the tolerances of kda_fwd hold for the
 * segment counts kda_fwd_cp_segments returns.
 * Errors: as kda_fwd_engine; KDA_ERR_INVALID_ARGUMENT for segments < 1 or
 * above 65536, KDA_ERR_WORKSPACE for a short workspace.
 */
kda_status_t kda_fwd_cp(const void *q, const void *k, const void *v,
                        const float *log_alpha, const float *beta, const float *S0,
                        const int32_t *cu_seqlens, int B, int T, int H, int d_k, int d_v,
                        int N, kda_dtype_t dtype, void *o, float *S_T, int segments,
                        void *workspace, size_t workspace_bytes, void *stream,
                        kda_engine_t engine);

/* Workspace bytes of kda_fwd_cp (0 for invalid sizes). */
size_t kda_fwd_cp_workspace_bytes(int N, int H, int d_k, int d_v, int segments);

/* A segment count for kda_fwd_cp on the current device: the smallest modelled
 * time with the first pass in one wave of N H (2 segments - 1) blocks over the
 * device's SMs; 1 (a plain kda_fwd) whenever N H already fills them.  Ttot is
 * the total number of tokens (the average sequence length sets the model). */
int kda_fwd_cp_segments(int N, int H, int64_t Ttot);

/* Largest N kda_fwd_noalloc accepts. */
#define KDA_NOALLOC_MAX_SEQS 16384

/*
 * kda_fwd_noalloc -- kda_fwd for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it is a convenience of
 * the library.  kda_fwd asks its caller for a workspace.  Callers that cannot
 * allocate -- code running where allocation is not allowed (a host callback on
 * a stream), a plugin inside a runtime that owns every device allocation, an
 * embedding without an allocator -- use this variant instead: it keeps the
 * scratch (status word and launch order) in a fixed 65,552-byte array in the
 * library's device memory, which every GPU that loads the library holds until
 * the process exits.  It calls no allocating routine.
 *
 * Arguments are those of kda_fwd without the workspace, plus `device_status`:
 * an optional (nullable, 4-byte aligned) device int32 that receives the
 * call's device status word (see kda_fwd) on `stream`.  The engine is chosen
 * as in kda_fwd.  N > KDA_NOALLOC_MAX_SEQS returns KDA_ERR_WORKSPACE before
 * anything is enqueued.
 *
 * The first call on a device looks up the scratch array's device address
 * (once per device, with that device current); make that first call before
 * any stream capture.  The address is kept with the id of the device's
 * context: after a cudaDeviceReset the next call looks it up again.  Every call shares the one array: calls that follow one
 * another are independent (each clears what must start at zero), but calls
 * that overlap on the GPU -- for example on two streams at once -- race.
 */
kda_status_t kda_fwd_noalloc(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta, const float *S0,
                             const int32_t *cu_seqlens, int B, int T, int H, int d_k, int d_v,
                             int N, kda_dtype_t dtype, void *o, float *S_T,
                             int32_t *device_status, void *stream);

/*
 * kda_decode_step -- one token for each of N sessions (the fused recurrent
 * form "完全拆解" recommends for decode, in its per-token order: decay,
 * old = Sbar^T k, S = Sbar + beta k (v - old)^T, o = S^T q).
 *
 *   q, k       [N, H, d_k] dtype      v, o  [N, H, d_v] dtype
 *   log_alpha  [N, H, d_k] fp32       beta  [N, H]      fp32
 *   S          [N, H, d_v, d_k] fp32, read and updated in place
 * Reads and writes the state exactly once.  No workspace.
 */
kda_status_t kda_decode_step(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta, float *S,
                             int N, int H, int d_k, int d_v, kda_dtype_t dtype,
                             void *o, void *stream);

/*
 * Output epilogue of a KDA layer, fused or as a pass of its own.
 *
 * After the recurrence, each head's output goes through a head-wise RMSNorm
 * over its d_v value channels and a sigmoid output gate, before the output
 * projection ("Kimi K3 模型结构（1）", output section: the norm runs per head
 * over the 128 channels and the sigmoid gate acts on every normalised channel;
 * "Kimi K3模型架构详解" section 3.2: y_t = W_o[Sigmoid(W_g x_t) . RMSNorm(o~_t)];
 * "完全拆解", the KDA layer).  Per (token, head):
 *
 *     y_v = sigmoid(g_v) * w_v * o_v / sqrt(mean_v'(o_v'^2) + eps)
 *
 * g holds the gate logits W_g x (the projection stays with the caller), w the
 * norm's per-channel weight, shared by all heads (NULL: ones), eps >= 0 the
 * norm's epsilon (with eps = 0 an all-zero o row gives NaN).  g and y have o's
 * layout and dtype.  The pages give neither eps nor where w lives; the
 * caller passes both.
 *
 * `mode` chooses where the epilogue runs: KDA_EPILOGUE_FUSED inside the
 * kernel's output stores (o never reaches HBM), KDA_EPILOGUE_SEPARATE as a
 * second pass (the kernel writes o into y, then kda_gated_rmsnorm runs on y
 * in place), KDA_EPILOGUE_AUTO the one measured faster on GB300: separate for
 * the prefill (its output stores sit on the latency-bound carry chain, where
 * the fused work costs more than the separate bandwidth-bound pass), fused for
 * the decode step.  Both give the same y up to rounding order.
 *
 * kda_fwd_gated: kda_fwd whose output is y instead of o.  g: [Ttot, H, d_v],
 * 16-byte aligned.  FUSED needs the tensor-core engine (KDA_ERR_UNSUPPORTED
 * otherwise).  Other arguments, engines, errors and device status as
 * kda_fwd_engine.
 * kda_decode_step_gated: kda_decode_step with the epilogue (g [N, H, d_v],
 * y [N, H, d_v]).
 * kda_gated_rmsnorm: the epilogue alone over `rows` rows of d_v channels
 * (rows = tokens x heads); o, g, y 16-byte aligned; y may alias o.
 */
typedef enum {
    KDA_EPILOGUE_AUTO = 0,
    KDA_EPILOGUE_FUSED = 1,
    KDA_EPILOGUE_SEPARATE = 2
} kda_epilogue_t;
kda_status_t kda_fwd_gated(const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta, const float *S0,
                           const int32_t *cu_seqlens, int B, int T, int H, int d_k, int d_v,
                           int N, kda_dtype_t dtype, const void *g, const float *norm_weight,
                           float eps, void *y, float *S_T, void *workspace,
                           size_t workspace_bytes, void *stream, kda_engine_t engine,
                           kda_epilogue_t mode);
kda_status_t kda_decode_step_gated(const void *q, const void *k, const void *v,
                                   const float *log_alpha, const float *beta, float *S,
                                   int N, int H, int d_k, int d_v, kda_dtype_t dtype,
                                   const void *g, const float *norm_weight, float eps,
                                   void *y, void *stream, kda_epilogue_t mode);
kda_status_t kda_gated_rmsnorm(const void *o, const void *g, const float *norm_weight,
                               float eps, int64_t rows, int d_v, kda_dtype_t dtype, void *y,
                               void *stream);

/*
 * Input prologue of a KDA layer ("Kimi Delta Attention 完全拆解", the KDA
 * layer's forward: q, k = L2Norm(Swish(ShortConv(W x))), v =
 * Swish(ShortConv(W_v x)); "Kimi K3 模型结构（1）", parameterisation section:
 * ShortConv is a depthwise causal convolution of kernel 4 along the sequence,
 * and decode keeps the last three projected inputs of q, k and v as the
 * layer's only state besides S).  Per stream, channel and token t:
 *
 *   c_t = w[0] x_{t-3} + w[1] x_{t-2} + w[2] x_{t-1} + w[3] x_t
 *   y_t = c_t * sigmoid(c_t)                                    (Swish)
 *   q_t, k_t = y_t / sqrt(sum over the d channels of y_t^2 + eps)  (per token, head;
 *              0 where that sum is 0);  v_t = y_t
 *
 * with x_{-3}, x_{-2}, x_{-1} of each sequence taken from the conv state.
 * Layout:
 *   xq, xk, xv  [Ttot, H, d] dtype: the projected inputs W x (16-byte aligned)
 *   wq, wk, wv  [H, d, 4] fp32 depthwise taps, w[3] on the current token
 *   conv        [N, 3, 3, H, d] fp32: per sequence (session) the three most
 *               recent inputs of stream q, k, v, oldest first
 *   q, k, v     [Ttot, H, d] dtype outputs
 *   d = 64 or 128; eps >= 0 finite.
 *
 * kda_short_conv: whole sequences (fixed length T, or packed with cu_seqlens as
 * in kda_fwd).  conv0 is the state before each sequence (NULL: zeros); conv_T
 * (NULL to skip) receives the state after it -- its last three inputs, with
 * conv0's tail for a sequence shorter than three -- and may alias conv0.  A
 * sequence run in pieces, each from the previous piece's conv_T, gives the
 * same outputs as one run.  workspace: at least kda_fwd_workspace_bytes(N)
 * bytes (the status word; a bad device-side cu_seqlens is reported as in
 * kda_fwd and nothing is written).
 * kda_short_conv_step: one token per session (xq, xk, xv, q, k, v [N, H, d]);
 * the state conv is read and moved on by one token in place.  No workspace.
 * Errors: KDA_ERR_INVALID_ARGUMENT for bad sizes, pointers or alignment,
 * KDA_ERR_UNSUPPORTED for other d, KDA_ERR_WORKSPACE for a short workspace.
 */
kda_status_t kda_short_conv(const void *xq, const void *xk, const void *xv, const float *wq,
                            const float *wk, const float *wv, const float *conv0,
                            const int32_t *cu_seqlens, int B, int T, int H, int d, int N,
                            kda_dtype_t dtype, float eps, void *q, void *k, void *v,
                            float *conv_T, void *workspace, size_t workspace_bytes,
                            void *stream);
kda_status_t kda_short_conv_step(const void *xq, const void *xk, const void *xv,
                                 const float *wq, const float *wk, const float *wv, float *conv,
                                 int N, int H, int d, kda_dtype_t dtype, float eps, void *q,
                                 void *k, void *v, void *stream);

/*
 * One decode token per session through the whole KDA layer step in one kernel
 * ("Kimi K3" (gentlecold) section 9.2: the inference kernel fuses the short
 * convolution, the input normalisation, the recurrence and the output
 * normalisation): the input prologue of kda_short_conv_step from the projected
 * inputs xq, xk, xv and the conv state, then the step of kda_decode_step, then
 * the epilogue of kda_decode_step_gated into y.  Layouts as there: xq, xk, xv,
 * g, y [N, H, d] dtype; wq, wk, wv [H, d, 4] fp32; conv [N, 3, 3, H, d] fp32 and
 * S [N, H, d, d] fp32, both updated in place; log_alpha [N, H, d], beta [N, H]
 * fp32; norm_weight [d] or NULL; l2_eps the prologue's L2Norm epsilon, eps the
 * RMSNorm's.  q, k and v stay in fp32 inside the kernel, so the result agrees
 * with the three separate calls up to the rounding of q, k, v to the io dtype.
 * Pointers 16-byte aligned.  No workspace.  Errors as kda_short_conv_step.
 */
kda_status_t kda_decode_layer_step(const void *xq, const void *xk, const void *xv,
                                   const float *wq, const float *wk, const float *wv, float *conv,
                                   float l2_eps, const float *log_alpha, const float *beta,
                                   float *S, int N, int H, int d, kda_dtype_t dtype,
                                   const void *g, const float *norm_weight, float eps, void *y,
                                   void *stream);

/*
 * Speculative-decode verification and commit ("Kimi K3 深度拆解" section 9.2:
 * the draft tokens' projected inputs are kept instead of a copy of the state
 * per draft position; after verification the accepted tokens are replayed on
 * chip and the resulting state is written back).  K draft tokens per session,
 * 1 <= K <= KDA_MAX_DRAFT_TOKENS:
 *
 *   q, k       [N, K, H, d_k] dtype      v, o  [N, K, H, d_v] dtype
 *   log_alpha  [N, K, H, d_k] fp32       beta  [N, K, H]      fp32
 *   S          [N, H, d_v, d_k] fp32
 *
 * kda_verify_tokens: o receives the outputs of the K tokens run in order from
 * S (token t sees the state after tokens 0 .. t); S is read once and not
 * written.  kda_commit_tokens: applies tokens 0 .. n_accept[n] - 1 of session
 * n to S in place (n_accept: device int32 [N], values clamped to [0, K];
 * NULL applies all K); S is read and written once.  Both agree with the same
 * tokens passed one at a time to kda_decode_step up to fp32 rounding (the
 * tokens are taken in closed form over sub-blocks of 8, which sums in another
 * order), except the outputs of a bf16 verify: it reads the state through bf16
 * products, so they agree to about the rounding of their own bf16 type.
 * Alignment as for kda_decode_step; n_accept 4-byte aligned.  No workspace.
 */
#define KDA_MAX_DRAFT_TOKENS 16
kda_status_t kda_verify_tokens(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, const float *S,
                               int N, int K, int H, int d_k, int d_v, kda_dtype_t dtype,
                               void *o, void *stream);
kda_status_t kda_commit_tokens(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, float *S,
                               const int32_t *n_accept, int N, int K, int H, int d_k, int d_v,
                               kda_dtype_t dtype, void *stream);

/* Synchronise `stream`, read the status word kda_fwd left in `workspace` and
 * return it (KDA_OK if no condition was raised).  KDA_ERR_CUDA if the copy or
 * the synchronisation fails. */
kda_status_t kda_read_device_status(const void *workspace, size_t workspace_bytes,
                                    void *stream);

/* Bytes of recurrent state for `layers` KDA layers, N sessions, H heads and
 * elem_bytes per element: layers * N * H * d_k * d_v * elem_bytes ("Kimi K3
 * 混合线性注意力" section 3: 69 x 96 x 128 x 128 x 2 B per session).
 * Returns 0 if any argument is negative or the product overflows. */
size_t kda_state_bytes(int layers, int N, int H, int d_k, int d_v, int elem_bytes);

/* Static, human-readable name of a status code. */
const char *kda_status_string(kda_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */

/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential fp64 CPU implementation of the Kimi Delta Attention
 * (KDA) recurrence.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  The GPU library shares no code, no
 * header and no constant with it; the product path never calls it.
 *
 * What it computes (per sequence n and head h, independently, t = 1..T):
 *
 *   alpha_t   = exp(log_alpha_t)                       (per key channel c)
 *   Sbar      = Diag(alpha_t) S_{t-1}                   decay
 *   old       = Sbar^T k_t                              response of the decayed state along k_t
 *   S_t       = Sbar + beta_t k_t (v_t - old)^T         erase + write (delta rule)
 *   o_t       = S_t^T q_t                               read from the UPDATED state
 *
 * This is the recurrence S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 * o_t = S_t^T q_t, taken in the five-step order that the pages spell out:
 *   - "Kimi K3 的 KDA" (marsggbo blog), section 3 (KDA: forget, erase, then write)
 *     and the single-head teaching loop of section 4;
 *   - "Kimi K3 ..." (gentlecold), section 3.2 (the KDA recurrence, decay first);
 *   - "Kimi Delta Attention 完全拆解" (pinghaoyang), the KDA equations with the
 *     decayed state S~ = Diag(alpha) S, and the per-token decode order listing
 *     (S_decay, old_value, S_t, memory_output).
 *
 * Logical state S[c][v] has key channel c in 0..dk-1 and value channel v in
 * 0..dv-1.  In memory it is stored transposed, mem[v*dk + c] = S[c][v]
 * (layout [N, H, d_v, d_k], the state layout the pages give for FlashKDA).
 *
 * The optional `erase = 0` mode drops the delta correction (old := 0), which is
 * the gated-linear-attention special case the pages use to explain chunking
 * ("Kimi K3 的 KDA", section 5; "完全拆解", degenerate cases).  It exists only
 * so that tests can check the pages' no-erase closed forms.
 *
 * The `plant` argument serves the test suite's mutation check.  Only a second,
 * test-only build of this file (compiled with -DKDA_ORACLE_PLANTS into
 * libkda_oracle_plants.so) contains planted mistakes: there a nonzero value
 * plants one deliberate, plausible slip so that the tests can show that the
 * pins catch it.  In the oracle proper, kda_token below is the method alone
 * and a nonzero `plant` is rejected.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One token for one (sequence, head): the five steps of the method.  S is the
 * [dv][dk] memory image (mem[v*dk + c] = S[c][v]); old is scratch of dv. */
static void kda_token(double *S, const double *q, const double *k, const double *v,
                      const double *g, double beta, int dk, int dv, int erase,
                      double *o, double *old)
{
    int c, j;

    /* step 1: decay each key channel c of the old state by alpha_c */
    for (j = 0; j < dv; ++j)
        for (c = 0; c < dk; ++c) S[(size_t)j * dk + c] *= exp(g[c]);

    /* step 2: old = Sbar^T k (the decayed state's answer along the current key) */
    for (j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (c = 0; c < dk; ++c) acc += S[(size_t)j * dk + c] * k[c];
        old[j] = erase ? acc : 0.0;
    }

    /* steps 3-4: erase the conflicting part along k, write the new value */
    for (j = 0; j < dv; ++j) {
        const double err = v[j] - old[j];
        for (c = 0; c < dk; ++c) S[(size_t)j * dk + c] += beta * k[c] * err;
    }

    /* step 5: read the updated state with the query */
    for (j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (c = 0; c < dk; ++c) acc += S[(size_t)j * dk + c] * q[c];
        o[j] = acc;
    }
}

#ifdef KDA_ORACLE_PLANTS
/* Test-only: the token step with one planted mistake (mutation check). */
enum {
    PLANT_NO_DECAY = 1,          /* alpha ignored */
    PLANT_ERASE_THEN_DECAY = 2,  /* (I - b k k^T) applied before Diag(alpha) */
    PLANT_ERASE_SIGN = 3,        /* v + old instead of v - old */
    PLANT_READ_BEFORE_WRITE = 4, /* o_t = Sbar^T q_t */
    PLANT_TRANSPOSED_OLD = 5,    /* old[v] = sum_c Sbar[v][c] k[c]  (needs dk == dv) */
    PLANT_DECAY_VALUE_AXIS = 6,  /* Diag(alpha) applied along v (needs dk == dv) */
    PLANT_BETA_ON_ERASE_ONLY = 7,/* write term without beta */
    PLANT_STALE_GATE = 8,        /* alpha of the previous token */
    PLANT_LAST = 8
};

static void planted_token(double *S, const double *q, const double *k, const double *v,
                          const double *g, const double *g_prev, double beta,
                          int dk, int dv, int erase, int plant, double *o, double *old)
{
    int c, j;
    const double *gate = (plant == PLANT_STALE_GATE) ? g_prev : g;

    if (plant == PLANT_ERASE_THEN_DECAY) {
        for (j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (c = 0; c < dk; ++c) acc += S[(size_t)j * dk + c] * k[c];
            old[j] = erase ? acc : 0.0;
        }
        for (j = 0; j < dv; ++j)
            for (c = 0; c < dk; ++c)
                S[(size_t)j * dk + c] = exp(gate[c]) *
                    (S[(size_t)j * dk + c] + beta * k[c] * (v[j] - old[j]));
        for (j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (c = 0; c < dk; ++c) acc += S[(size_t)j * dk + c] * q[c];
            o[j] = acc;
        }
        return;
    }
    if (plant != PLANT_NO_DECAY) {
        for (j = 0; j < dv; ++j)
            for (c = 0; c < dk; ++c) {
                double a = (plant == PLANT_DECAY_VALUE_AXIS) ? exp(gate[j]) : exp(gate[c]);
                S[(size_t)j * dk + c] *= a;
            }
    }
    if (plant == PLANT_READ_BEFORE_WRITE) {
        for (j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (c = 0; c < dk; ++c) acc += S[(size_t)j * dk + c] * q[c];
            o[j] = acc;
        }
    }
    for (j = 0; j < dv; ++j) {
        double acc = 0.0;
        if (plant == PLANT_TRANSPOSED_OLD) {
            for (c = 0; c < dk; ++c) acc += S[(size_t)c * dk + j] * k[c];
        } else {
            for (c = 0; c < dk; ++c) acc += S[(size_t)j * dk + c] * k[c];
        }
        old[j] = erase ? acc : 0.0;
    }
    for (j = 0; j < dv; ++j) {
        const double err = (plant == PLANT_ERASE_SIGN) ? v[j] + old[j] : v[j] - old[j];
        for (c = 0; c < dk; ++c) {
            const double upd = (plant == PLANT_BETA_ON_ERASE_ONLY)
                                   ? k[c] * v[j] - beta * k[c] * old[j]
                                   : beta * k[c] * err;
            S[(size_t)j * dk + c] += upd;
        }
    }
    if (plant != PLANT_READ_BEFORE_WRITE) {
        for (j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (c = 0; c < dk; ++c) acc += S[(size_t)j * dk + c] * q[c];
            o[j] = acc;
        }
    }
}
#else
enum { PLANT_LAST = 0 };
#endif

/*
 * Forward over packed sequences.
 *   q, log_alpha : [Ttot][H][dk]      k : [Ttot][H][dk]      v : [Ttot][H][dv]
 *   beta         : [Ttot][H]
 *   S0           : [N][H][dv][dk] or NULL (zero initial state)
 *   cu_seqlens   : [N+1] token offsets, cu_seqlens[0] = 0, non-decreasing
 *   o            : [Ttot][H][dv]     S_T : [N][H][dv][dk] or NULL
 * Returns 0, or -1 on a bad argument.
 */
int kda_oracle_fwd(const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *beta, const double *S0,
                   const int64_t *cu_seqlens, int N, int H, int dk, int dv,
                   int erase, int plant, double *o, double *S_T)
{
    long long p;
    int bad = 0;
    if (!q || !k || !v || !log_alpha || !beta || !cu_seqlens || !o) return -1;
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (plant < 0 || plant > PLANT_LAST) return -1;
#ifdef KDA_ORACLE_PLANTS
    if ((plant == PLANT_TRANSPOSED_OLD || plant == PLANT_DECAY_VALUE_AXIS) && dk != dv) return -1;
#endif
    if (cu_seqlens[0] != 0) return -1;
    for (p = 0; p < N; ++p)
        if (cu_seqlens[p + 1] < cu_seqlens[p]) return -1;

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (p = 0; p < (long long)N * H; ++p) {
        const int n = (int)(p / H), h = (int)(p % H);
        const size_t state = (size_t)dk * dv;
        double *S = (double *)malloc(sizeof(double) * (state + dv + dk));
        double *old, *zero_gate;
        int64_t t;
        if (!S) { bad |= 1; continue; }
        old = S + state;
        zero_gate = old + dv;
        memset(zero_gate, 0, sizeof(double) * dk);
        if (S0) memcpy(S, S0 + ((size_t)n * H + h) * state, sizeof(double) * state);
        else memset(S, 0, sizeof(double) * state);
        for (t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            const size_t row = (size_t)t * H + h;
#ifdef KDA_ORACLE_PLANTS
            if (plant) {
                const double *g_prev = (t > cu_seqlens[n]) ? log_alpha + (row - H) * dk : zero_gate;
                planted_token(S, q + row * dk, k + row * dk, v + row * dv, log_alpha + row * dk,
                              g_prev, beta[row], dk, dv, erase, plant, o + row * dv, old);
                continue;
            }
#endif
            kda_token(S, q + row * dk, k + row * dk, v + row * dv, log_alpha + row * dk,
                      beta[row], dk, dv, erase, o + row * dv, old);
        }
        if (S_T) memcpy(S_T + ((size_t)n * H + h) * state, S, sizeof(double) * state);
        free(S);
    }
    return bad ? -1 : 0;
}

/*
 * One decode step for N sessions: the same token update applied once per
 * (session, head), continuing from S in place.
 *   q, k, log_alpha : [N][H][dk]   v, o : [N][H][dv]   beta : [N][H]
 *   S               : [N][H][dv][dk], updated in place
 */
int kda_oracle_decode_step(const double *q, const double *k, const double *v,
                           const double *log_alpha, const double *beta, double *S,
                           int N, int H, int dk, int dv, double *o)
{
    long long p;
    int bad = 0;
    if (!q || !k || !v || !log_alpha || !beta || !S || !o) return -1;
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (p = 0; p < (long long)N * H; ++p) {
        double *old = (double *)malloc(sizeof(double) * dv);
        if (!old) { bad |= 1; continue; }
        kda_token(S + (size_t)p * dk * dv, q + (size_t)p * dk, k + (size_t)p * dk,
                  v + (size_t)p * dv, log_alpha + (size_t)p * dk, beta[p], dk, dv, 1,
                  o + (size_t)p * dv, old);
        free(old);
    }
    return bad ? -1 : 0;
}

/* Threads OpenMP will use (reported with the CPU baseline). */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

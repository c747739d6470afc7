/*
 * kda_oracle.c -- plain fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * links, includes or calls it, and it shares no code with the CUDA path.
 *
 * What it computes.  The pages name KDA's objects -- BF16 Q/K/V with an FP32
 * recurrent state (cuLA PR #110, "feat(cp): add opt-in NVSHMEM CP state
 * handoff", §Supported configuration), an affine recurrence state per shard
 * (same page, §Motivation), and a transition plus a state update per shard
 * (cuLA PR #136, "feat(kda): add cuDNN concatenated-summary Kimi CP",
 * §Summary) -- but never write the equations.  This file uses the KDA gated
 * delta rule with a K x V state (non-transposed layout, PR #110 §Supported
 * configuration), a per-key-channel log-decay g_t, and a per-token beta_t:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * taken token by token exactly as written: first the decay, then the
 * delta-rule correction against the decayed state, then the output from the
 * updated state.  Inputs arrive as the exact fp32 values of the bf16 / fp32
 * tensors; every operation is done in double with the C library's exp().
 *
 * The "transition" of a token range is the same recurrence run on a K x K
 * matrix P with zero values (the homogeneous part), started from the identity:
 *     P_t = (I - beta_t k_t k_t^T) Diag(exp g_t) P_{t-1}.
 * Then the state after the range is P_end S_start + S_end|_{S_start = 0}, and
 * the query seen through the transition is qhat_t = scale * P_t^T q_t.
 *
 * The 'mutate' argument exists only so that tests can plant a plausible mistake
 * in the oracle and check that the pins catch it; every caller other than
 * those tests passes 0.
 *
 * Layouts (row-major, contiguous): q,k,g [T][H][K]; v [T][H][V]; beta [T][H];
 * states [K][V]; transitions [K][K]; o [T][H][V].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    MUT_NONE = 0,
    MUT_DECAY_AFTER_DELTA = 1,   /* decay applied after the delta-rule correction */
    MUT_OUTPUT_OLD_STATE = 2,    /* o_t read from S_{t-1} instead of S_t */
    MUT_OUTPUT_TRANSPOSED = 3,   /* o_t = S_t q_t instead of S_t^T q_t */
    MUT_PROJECT_UNDECAYED = 4,   /* correction projects the undecayed S_{t-1} */
    MUT_DECAY_SIGN = 5,          /* exp(-g) instead of exp(g) */
    MUT_DROP_BETA = 6,           /* beta dropped from the correction */
    MUT_DECAY_ON_VALUE_AXIS = 7  /* decay scales the value columns, not key rows */
};

/* One token of the recurrence on an R x W matrix X (R = K rows indexed by the
 * key channel, W columns).  val (length W) is v_t for the state and NULL for
 * the homogeneous transition.  tmp has room for W doubles. */
static void token_step(double *X, int R, int W, const float *k, const float *g, double beta,
                       const float *val, double *tmp, int mutate)
{
    int i, j;
    if (mutate != MUT_DECAY_AFTER_DELTA && mutate != MUT_PROJECT_UNDECAYED) {
        for (i = 0; i < R; ++i) {
            double d = exp(mutate == MUT_DECAY_SIGN ? -(double)g[i] : (double)g[i]);
            for (j = 0; j < W; ++j) {
                double dj = (mutate == MUT_DECAY_ON_VALUE_AXIS && j < R) ? exp((double)g[j]) : d;
                X[(size_t)i * W + j] *= dj;
            }
        }
    }
    /* tmp = X^T k  (projection of the decayed state on the key) */
    for (j = 0; j < W; ++j) tmp[j] = 0.0;
    for (i = 0; i < R; ++i) {
        double ki = (double)k[i];
        for (j = 0; j < W; ++j) tmp[j] += X[(size_t)i * W + j] * ki;
    }
    if (mutate == MUT_PROJECT_UNDECAYED) {
        for (i = 0; i < R; ++i) {
            double d = exp((double)g[i]);
            for (j = 0; j < W; ++j) X[(size_t)i * W + j] *= d;
        }
    }
    /* X += beta k (val - X^T k)^T */
    double b = (mutate == MUT_DROP_BETA) ? 1.0 : beta;
    for (i = 0; i < R; ++i) {
        double bk = b * (double)k[i];
        for (j = 0; j < W; ++j) {
            double target = val ? (double)val[j] : 0.0;
            X[(size_t)i * W + j] += bk * (target - tmp[j]);
        }
    }
    if (mutate == MUT_DECAY_AFTER_DELTA) {
        for (i = 0; i < R; ++i) {
            double d = exp((double)g[i]);
            for (j = 0; j < W; ++j) X[(size_t)i * W + j] *= d;
        }
    }
}

/* out[j] = scale * sum_i X[i][j] q[i]  (X^T q), or X q under the transposed mutation. */
static void read_out(const double *X, int R, int W, const float *q, double scale, double *out, int mutate)
{
    int i, j;
    if (mutate == MUT_OUTPUT_TRANSPOSED && R == W) {
        for (i = 0; i < R; ++i) {
            double acc = 0.0;
            for (j = 0; j < W; ++j) acc += X[(size_t)i * W + j] * (double)q[j];
            out[i] = scale * acc;
        }
        return;
    }
    for (j = 0; j < W; ++j) out[j] = 0.0;
    for (i = 0; i < R; ++i) {
        double qi = (double)q[i];
        for (j = 0; j < W; ++j) out[j] += X[(size_t)i * W + j] * qi;
    }
    for (j = 0; j < W; ++j) out[j] *= scale;
}

/*
 * Run tokens [t0, t1) of head h.
 *   S     [K][V] in/out: state at t0 on entry, state at t1 on exit (may be NULL)
 *   P     [K][K] in/out: transition on entry (callers pass I), on exit (may be NULL)
 *   o     [(t1-t0)][V] out: scale * S_t^T q_t (may be NULL; needs S)
 *   qhat  [(t1-t0)][K] out: scale * P_t^T q_t (may be NULL; needs P)
 * Returns 0, or -1 on a bad argument.
 */
int oracle_kda_run(int64_t t0, int64_t t1, int32_t h, int32_t H, int32_t K, int32_t V,
                   const float *q, const float *k, const float *v, const float *g,
                   const float *beta, double scale, double *S, double *P,
                   double *o, double *qhat, int mutate)
{
    if (t1 < t0 || h < 0 || h >= H || K <= 0 || V <= 0) return -1;
    if ((o && !S) || (qhat && !P)) return -1;
    int W = V > K ? V : K;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)W);
    double *prev = NULL;
    if (!tmp) return -1;
    if (mutate == MUT_OUTPUT_OLD_STATE) {
        prev = (double *)malloc(sizeof(double) * (size_t)K * (size_t)W);
        if (!prev) { free(tmp); return -1; }
    }
    for (int64_t t = t0; t < t1; ++t) {
        size_t qk_off = ((size_t)t * H + h) * (size_t)K;
        size_t v_off = ((size_t)t * H + h) * (size_t)V;
        const float *kt = k + qk_off;
        const float *gt = g + qk_off;
        const float *qt = q + qk_off;
        double bt = (double)beta[(size_t)t * H + h];
        if (S) {
            if (prev) memcpy(prev, S, sizeof(double) * (size_t)K * V);
            token_step(S, K, V, kt, gt, bt, v + v_off, tmp, mutate);
            if (o) read_out(prev ? prev : S, K, V, qt, scale, o + (size_t)(t - t0) * V, mutate);
        }
        if (P) {
            if (prev) memcpy(prev, P, sizeof(double) * (size_t)K * K);
            token_step(P, K, K, kt, gt, bt, NULL, tmp, mutate);
            if (qhat) read_out(prev ? prev : P, K, K, qt, scale, qhat + (size_t)(t - t0) * K, mutate);
        }
    }
    free(prev);
    free(tmp);
    return 0;
}

/*
 * Monolithic forward over packed sequences: for every (sequence n, head h)
 * the state starts at h0[n][h] (zeros when h0 is NULL) at the sequence's first
 * token and runs to its last token.  o: [T][H][V] (NULL to skip),
 * final_state: [N][H][K][V] (NULL to skip).  Heads listed in 'heads'
 * (length n_heads) are computed; pass heads = NULL for all H.
 * Parallel over (sequence, head) with OpenMP using 'nthreads' threads
 * (<= 0: the OpenMP default).
 */
int oracle_kda_forward(int32_t N, const int32_t *cu_seqlens, int32_t H, int32_t K, int32_t V,
                       const float *q, const float *k, const float *v, const float *g,
                       const float *beta, const double *h0, double scale,
                       const int32_t *heads, int32_t n_heads,
                       double *o, double *final_state, int nthreads, int mutate)
{
    if (N <= 0 || H <= 0 || K <= 0 || V <= 0 || !cu_seqlens) return -1;
    for (int32_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    int32_t nh = heads ? n_heads : H;
    int64_t tasks = (int64_t)N * nh;
    int err = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : err)
#endif
    for (int64_t task = 0; task < tasks; ++task) {
        int32_t n = (int32_t)(task / nh);
        int32_t h = heads ? heads[task % nh] : (int32_t)(task % nh);
        if (h < 0 || h >= H) { err |= 1; continue; }
        size_t kv = (size_t)K * V;
        double *S = (double *)malloc(sizeof(double) * kv);
        double *ob = NULL;
        int64_t t0 = cu_seqlens[n], t1 = cu_seqlens[n + 1];
        if (!S) { err |= 1; continue; }
        if (h0) memcpy(S, h0 + ((size_t)n * H + h) * kv, sizeof(double) * kv);
        else memset(S, 0, sizeof(double) * kv);
        if (o && t1 > t0) {
            ob = (double *)malloc(sizeof(double) * (size_t)(t1 - t0) * V);
            if (!ob) { free(S); err |= 1; continue; }
        }
        if (oracle_kda_run(t0, t1, h, H, K, V, q, k, v, g, beta, scale, S, NULL, ob, NULL, mutate) != 0)
            err |= 1;
        if (ob) {
            for (int64_t t = t0; t < t1; ++t)
                memcpy(o + ((size_t)t * H + h) * V, ob + (size_t)(t - t0) * V, sizeof(double) * V);
            free(ob);
        }
        if (final_state) memcpy(final_state + ((size_t)n * H + h) * kv, S, sizeof(double) * kv);
        free(S);
    }
    return err ? -1 : 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * KDA chunked-prefill ORACLE -- test infrastructure only.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  The product path (libkda.so and its Python
 * binding) never calls it and shares no code, header or constant with it.
 *
 * What it computes: the bounded-gate KDA recurrence, token by token, in
 * IEEE double precision, one (sequence, head) pair at a time.  This is the
 * plain definition of the operation, with no chunking, blocking or
 * reordering.  Sources (vLLM PR reports on prhub.com.cn):
 *
 *   - "[Perf][GLM-5.3-Flash] Use FlashKDA for KDA chunked prefill"
 *     (PR #55737), Features & motivation and Implementation breakdown
 *     item 3: the kernel takes raw gate logits g and raw beta logits,
 *     l2-normalises q and k itself, and applies the bounded gate
 *     lower_bound * sigmoid(exp(A_log) * (g + dt_bias)); scale is
 *     head_dim**-0.5 and is applied to q; A_log is one value per head,
 *     dt_bias is [heads, head_dim]; sequences are packed by cu_seqlens;
 *     initial_state in, final_state out, shaped (seqs, heads, 128, 128).
 *   - "[KDA] Update flashKDA to support bf16 checkpoint state"
 *     (PR #56485), Implementation breakdown item 2: the state may be
 *     stored in fp32 or bf16 (storage rounding is the caller's business
 *     here: the oracle reads and writes doubles).
 *
 * Readings where the pages are silent (each also listed in the design
 * notes): the gate value a = lb*sigmoid(...) is a per-key-channel LOG decay
 * (lb <= 0, so a lies in (lb, 0]); the state S is Dk x Dv, row = key
 * channel, column = value channel; per token the state is first decayed,
 * then receives the delta-rule write, then is read with q (read after
 * write); beta = sigmoid(raw beta logit); l2norm is x / sqrt(sum x^2 + eps).
 *
 * Per token t of sequence n, head h (vectors are length D):
 *   qh = q_t / sqrt(|q_t|^2 + eps)          kh = k_t / sqrt(|k_t|^2 + eps)
 *   a  = lb * sigmoid(exp(A_log[h]) * (g_t + dt_bias[h,:]))
 *   S  = diag(exp(a)) S                      (rows = key channels decay)
 *   b  = sigmoid(beta_logit_t)
 *   u  = b * (v_t - S^T kh)                  (delta-rule correction)
 *   S  = S + kh u^T
 *   o_t = scale * S^T qh
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }

/* One (sequence, head) pair.  S is D*D doubles, read as the initial state
 * and left holding the final state.  Work vectors: 5*D doubles. */
static void recur_one(int64_t t0, int64_t t1, int h, int H, int D,
                      const double* q, const double* k, const double* v,
                      const double* g, const double* beta_logit,
                      double A_log_h, const double* dt_bias_h,
                      double lower_bound, double scale, double eps,
                      double* S, double* out, double* work)
{
    double* qh = work;
    double* kh = work + D;
    double* decay = work + 2 * D;
    double* u = work + 3 * D;
    double* o = work + 4 * D;
    const double gate_scale = exp(A_log_h);

    for (int64_t t = t0; t < t1; ++t) {
        const int64_t row = (t * H + h) * (int64_t)D;
        const double* qt = q + row;
        const double* kt = k + row;
        const double* vt = v + row;
        const double* gt = g + row;

        /* l2 normalisation of q and k, then scale on q */
        double sq = 0.0, sk = 0.0;
        for (int d = 0; d < D; ++d) {
            sq += qt[d] * qt[d];
            sk += kt[d] * kt[d];
        }
        const double iq = 1.0 / sqrt(sq + eps);
        const double ik = 1.0 / sqrt(sk + eps);
        for (int d = 0; d < D; ++d) {
            qh[d] = qt[d] * iq * scale;
            kh[d] = kt[d] * ik;
        }

        /* bounded gate: per-key-channel log decay a in (lb, 0] */
        for (int d = 0; d < D; ++d) {
            const double a = lower_bound * sigmoid_d(gate_scale * (gt[d] + dt_bias_h[d]));
            decay[d] = exp(a);
        }

        /* decay the rows of S */
        for (int d = 0; d < D; ++d)
            for (int c = 0; c < D; ++c)
                S[d * D + c] *= decay[d];

        /* delta-rule write: u = beta * (v - S^T kh); S += kh u^T */
        const double b = sigmoid_d(beta_logit[t * H + h]);
        for (int c = 0; c < D; ++c) u[c] = 0.0;
        for (int d = 0; d < D; ++d)
            for (int c = 0; c < D; ++c)
                u[c] += S[d * D + c] * kh[d];
        for (int c = 0; c < D; ++c) u[c] = b * (vt[c] - u[c]);
        for (int d = 0; d < D; ++d)
            for (int c = 0; c < D; ++c)
                S[d * D + c] += kh[d] * u[c];

        /* read after the write: o = S^T (scale * qh) */
        for (int c = 0; c < D; ++c) o[c] = 0.0;
        for (int d = 0; d < D; ++d)
            for (int c = 0; c < D; ++c)
                o[c] += S[d * D + c] * qh[d];
        for (int c = 0; c < D; ++c) out[row + c] = o[c];
    }
}

/*
 * Layouts (all row-major, all doubles except cu_seqlens):
 *   q, k, v, g   [T][H][D]          beta_logit [T][H]
 *   A_log        [H]                dt_bias    [H][D]
 *   initial_state, final_state [N][H][D][D]  (key channel major)
 *   cu_seqlens   [N+1] int32, 0 = cu[0] <= cu[1] <= ... <= cu[N] <= T
 *   out          [T][H][D]  (rows of tokens past cu[N] are not written)
 * initial_state may be NULL (zero state).  Returns 0, or -1 on bad
 * arguments.  num_threads <= 0 means the OpenMP default.
 */
int kda_oracle_fwd(int64_t T, int32_t N, int32_t H, int32_t D,
                   const double* q, const double* k, const double* v,
                   const double* g, const double* beta_logit,
                   const double* A_log, const double* dt_bias,
                   double lower_bound, double scale, double eps,
                   const double* initial_state, const int32_t* cu_seqlens,
                   double* out, double* final_state, int num_threads)
{
    if (T < 0 || N < 0 || H <= 0 || D <= 0) return -1;
    if (!q || !k || !v || !g || !beta_logit || !A_log || !dt_bias) return -1;
    if (!cu_seqlens || !out || !final_state) return -1;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] > T) return -1;
    for (int32_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;

    const int64_t pairs = (int64_t)N * H;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
    {
        /* every thread reaches the worksharing loop, even if its allocation
         * failed: it then only records the failure */
        double* work = (double*)malloc(sizeof(double) * 5 * (size_t)D);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t p = 0; p < pairs; ++p) {
            if (!work) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                failed = 1;
                continue;
            }
            const int32_t n = (int32_t)(p / H);
            const int h = (int)(p % H);
            double* S = final_state + p * (int64_t)D * D;
            if (initial_state)
                memcpy(S, initial_state + p * (int64_t)D * D, sizeof(double) * (size_t)D * D);
            else
                memset(S, 0, sizeof(double) * (size_t)D * D);
            recur_one(cu_seqlens[n], cu_seqlens[n + 1], h, H, D, q, k, v, g,
                      beta_logit, A_log[h], dt_bias + (int64_t)h * D,
                      lower_bound, scale, eps, S, out, work);
        }
        free(work);
    }
    return failed ? -1 : 0;
}

/* Number of threads the OpenMP runtime would use (1 without OpenMP). */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

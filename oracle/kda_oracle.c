/*
 * KDA oracle: plain, sequential, fp64 CPU implementation of the Kimi Delta
 * Attention recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline arm may load this library.  It shares no code, header or
 * constant with the CUDA path and must never be called by it.
 *
 * What it computes (Wikipedia-mirror page "Kimi (AI)", section "Kimi Delta
 * Attention (KDA)", the three-line update block after the naive linear
 * attention equation):
 *
 *     S~_t = diag(alpha_t) S_{t-1}                  (forget gating)
 *     v~_t = S~_t k_t                               (predict)
 *     S_t  = S~_t + beta_t (v_t - v~_t) k_t^T       (memory updating)
 *
 * and the output read from the naive linear attention line of the same
 * section, o_t = S_t q_t, applied to KDA's S_t (the post-update state).
 *
 * S is d_v x d_k because the page builds it as a sum of v k^T outer products;
 * diag(alpha_t) multiplies from the left, so alpha_t has d_v entries and
 * scales the rows (value channels).  beta_t is one scalar per token and head.
 * No softmax scale, normalisation or output gate: none appears on the page.
 *
 * Each step is written out literally, in the order the page gives it, with
 * no chunking, blocking or reordering.  Inputs arrive in their storage types
 * (bf16 bit patterns or fp32) and are widened exactly to fp64.  Build flags:
 * -O2 -ffp-contract=off, never -ffast-math.
 *
 * Layouts (row-major, last index fastest):
 *   q, k       [T_total][H][d_k]     kind 0: bf16 bits (uint16), kind 1: fp32
 *   v          [T_total][H][d_v]     same kind as q, k
 *   alpha      [T_total][H][d_v]     fp32
 *   beta       [T_total][H]          fp32
 *   S0         [N][H][d_v][d_k]      fp64, or NULL for zeros
 *   cu_seqlens [N+1]                 int32, cu[0] = 0, non-decreasing
 *   o          [T_total][H][d_v]     fp64 output
 *   S_T        [N][H][d_v][d_k]      fp64 output (may be NULL)
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Widen a bf16 bit pattern: it is the upper half of an IEEE binary32. */
static double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double oracle_load(const void* base, int kind, int64_t idx)
{
    if (kind == 0) return oracle_bf16_to_f64(((const uint16_t*)base)[idx]);
    return (double)((const float*)base)[idx];
}

/* One (sequence, head) pair, all of its tokens in order. */
static void oracle_run_pair(const void* q, const void* k, const void* v, int kind,
                            const float* alpha, const float* beta, const double* S0,
                            int64_t t_begin, int64_t t_end, int32_t n, int32_t h,
                            int32_t H, int32_t d_k, int32_t d_v,
                            double* o, double* S_T,
                            double* S, double* kt, double* qt, double* vpred)
{
    const int64_t state_off = ((int64_t)n * H + h) * (int64_t)d_v * d_k;
    if (S0) memcpy(S, S0 + state_off, sizeof(double) * (size_t)d_v * d_k);
    else memset(S, 0, sizeof(double) * (size_t)d_v * d_k);

    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t th = t * H + h;
        for (int32_t c = 0; c < d_k; ++c) {
            kt[c] = oracle_load(k, kind, th * d_k + c);
            qt[c] = oracle_load(q, kind, th * d_k + c);
        }
        const double b = (double)beta[th];

        /* forget gating: S~ = diag(alpha_t) S_{t-1}; row r scaled by alpha_t[r] */
        for (int32_t r = 0; r < d_v; ++r) {
            const double a = (double)alpha[th * d_v + r];
            double* row = S + (int64_t)r * d_k;
            for (int32_t c = 0; c < d_k; ++c) row[c] = a * row[c];
        }
        /* predict: v~ = S~ k_t */
        for (int32_t r = 0; r < d_v; ++r) {
            const double* row = S + (int64_t)r * d_k;
            double acc = 0.0;
            for (int32_t c = 0; c < d_k; ++c) acc += row[c] * kt[c];
            vpred[r] = acc;
        }
        /* memory updating: S = S~ + beta_t (v_t - v~) k_t^T */
        for (int32_t r = 0; r < d_v; ++r) {
            const double err = oracle_load(v, kind, th * d_v + r) - vpred[r];
            double* row = S + (int64_t)r * d_k;
            for (int32_t c = 0; c < d_k; ++c) row[c] = row[c] + b * err * kt[c];
        }
        /* output: o_t = S_t q_t */
        for (int32_t r = 0; r < d_v; ++r) {
            const double* row = S + (int64_t)r * d_k;
            double acc = 0.0;
            for (int32_t c = 0; c < d_k; ++c) acc += row[c] * qt[c];
            o[th * d_v + r] = acc;
        }
    }
    if (S_T) memcpy(S_T + state_off, S, sizeof(double) * (size_t)d_v * d_k);
}

/*
 * Runs every (sequence, head) pair of a packed batch.  Returns 0 on success,
 * 1 on bad sizes, 2 on a cu_seqlens that does not start at 0, decreases, or
 * ends past total_tokens, 3 when scratch memory cannot be allocated.  Pairs
 * run in parallel over `nthreads` OpenMP threads (<= 0: library default);
 * the arithmetic of each pair is sequential and does not depend on it.
 */
int kda_oracle_prefill(const void* q, const void* k, const void* v, int kind,
                       const float* alpha, const float* beta, const double* S0,
                       const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                       int32_t H, int32_t d_k, int32_t d_v,
                       double* o, double* S_T, int32_t nthreads)
{
    if (num_seqs < 0 || H <= 0 || d_k <= 0 || d_v <= 0 || (kind != 0 && kind != 1)) return 1;
    if (!cu_seqlens || (num_seqs > 0 && (!q || !k || !v || !alpha || !beta || !o))) return 1;
    if (cu_seqlens[0] != 0) return 2;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
    if ((int64_t)cu_seqlens[num_seqs] > total_tokens) return 2;

    const int64_t pairs = (int64_t)num_seqs * H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(|: failed)
#endif
    {
        double* S = (double*)malloc(sizeof(double) * (size_t)d_v * d_k);
        double* kt = (double*)malloc(sizeof(double) * (size_t)d_k);
        double* qt = (double*)malloc(sizeof(double) * (size_t)d_k);
        double* vpred = (double*)malloc(sizeof(double) * (size_t)d_v);
        const int have_scratch = S && kt && qt && vpred;
        if (!have_scratch) failed = 1;
        /* every thread reaches the work-sharing loop; one without scratch skips its pairs */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t p = 0; p < pairs; ++p) {
            if (!have_scratch) continue;
            const int32_t n = (int32_t)(p / H), h = (int32_t)(p % H);
            oracle_run_pair(q, k, v, kind, alpha, beta, S0, cu_seqlens[n], cu_seqlens[n + 1],
                            n, h, H, d_k, d_v, o, S_T, S, kt, qt, vpred);
        }
        free(S); free(kt); free(qt); free(vpred);
    }
    return failed ? 3 : 0;
}

/* Number of OpenMP threads a call with nthreads <= 0 would use. */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

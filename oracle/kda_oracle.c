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
                            int32_t H, int32_t d_k, int32_t d_v, int additive,
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
        /* predict: v~ = S~ k_t (none in the additive update of linear attention) */
        for (int32_t r = 0; r < d_v && additive; ++r) vpred[r] = 0.0;
        for (int32_t r = 0; r < d_v && !additive; ++r) {
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
static int oracle_prefill_rule(const void* q, const void* k, const void* v, int kind,
                               const float* alpha, const float* beta, const double* S0,
                               const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                               int32_t H, int32_t d_k, int32_t d_v, int additive,
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
                            n, h, H, d_k, d_v, additive, o, S_T, S, kt, qt, vpred);
        }
        free(S); free(kt); free(qt); free(vpred);
    }
    return failed ? 3 : 0;
}

/* The KDA recurrence over a packed batch (the delta rule). */
int kda_oracle_prefill(const void* q, const void* k, const void* v, int kind,
                       const float* alpha, const float* beta, const double* S0,
                       const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                       int32_t H, int32_t d_k, int32_t d_v,
                       double* o, double* S_T, int32_t nthreads)
{
    return oracle_prefill_rule(q, k, v, kind, alpha, beta, S0, cu_seqlens, num_seqs,
                               total_tokens, H, d_k, d_v, 0, o, S_T, nthreads);
}

/*
 * The same recurrence with the additive update of linear attention instead of
 * the delta rule: predict is dropped (v~ = 0), so S_t = diag(alpha_t) S_{t-1}
 * + beta_t v_t k_t^T and o_t = S_t q_t.  With alpha = beta = 1 it is the
 * page's naive linear attention, S_t = S_{t-1} + v_t k_t^T ("Kimi (AI)",
 * section "Kimi Delta Attention (KDA)", the line before the three-line
 * update).  Same arguments and return codes as kda_oracle_prefill.
 */
int kda_oracle_prefill_additive(const void* q, const void* k, const void* v, int kind,
                                const float* alpha, const float* beta, const double* S0,
                                const int32_t* cu_seqlens, int32_t num_seqs,
                                int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                double* o, double* S_T, int32_t nthreads)
{
    return oracle_prefill_rule(q, k, v, kind, alpha, beta, S0, cu_seqlens, num_seqs,
                               total_tokens, H, d_k, d_v, 1, o, S_T, nthreads);
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

/*
 * ---------------------------------------------------------------------------
 * Reverse mode of the same recurrence (gradients for training).
 *
 * The pages place the chunk-wise parallel form in training, which needs the
 * gradients of a loss L with respect to every input.  Given dL/do_t and
 * dL/dS_T, the chain rule through the three-line update taken backwards
 * (memory updating, predict, forget gating, in that order) gives, with
 * D = dL/dS_t accumulated from the later tokens and u = v_t - v~_t:
 *
 *     D       += do_t q_t^T                    (o_t = S_t q_t)
 *     dq_t     = S_t^T do_t
 *     g        = D k_t
 *     dv_t     = beta_t g
 *     dbeta_t  = u^T g
 *     dk_t     = beta_t (D^T u - S~_t^T g)
 *     dS~      = D - beta_t g k_t^T
 *     dalpha_t = rowwise sum of dS~ (*) S_{t-1}
 *     D        = diag(alpha_t) dS~             (dL/dS_{t-1})
 *
 * and dL/dS0 is the D left after the first token.  The states S_{t-1} are
 * taken from a plain tape: the forward pass keeps every OR_SEG-th state, and
 * the backward pass re-runs the forward step from the nearest kept state to
 * refill the states of one segment at a time.  Re-running the same fp64
 * step gives the same states bit for bit, so the tape only bounds memory.
 * ---------------------------------------------------------------------------
 */
#define OR_SEG 64

/* One forward step of one (sequence, head): S_prev -> S_next (the forget gating,
 * predict and memory updating lines above, written out once more). */
static void oracle_step(const double* S_prev, double* S_next, const double* kt,
                        const double* vt, const double* at, double b, int32_t d_k,
                        int32_t d_v)
{
    for (int32_t r = 0; r < d_v; ++r) {
        const double* src = S_prev + (int64_t)r * d_k;
        double* row = S_next + (int64_t)r * d_k;
        for (int32_t c = 0; c < d_k; ++c) row[c] = at[r] * src[c];      /* S~ */
        double pred = 0.0;
        for (int32_t c = 0; c < d_k; ++c) pred += row[c] * kt[c];       /* v~ */
        const double err = vt[r] - pred;
        for (int32_t c = 0; c < d_k; ++c) row[c] += b * err * kt[c];
    }
}

typedef struct {
    double *tape, *kt, *qt, *vt, *at, *dot, *D, *Stl, *g, *u;
} oracle_bwd_scratch;

static void oracle_load_token(const void* q, const void* k, const void* v, int kind,
                              const float* alpha, int64_t th, int32_t d_k, int32_t d_v,
                              double* qt, double* kt, double* vt, double* at)
{
    for (int32_t c = 0; c < d_k; ++c) {
        qt[c] = oracle_load(q, kind, th * d_k + c);
        kt[c] = oracle_load(k, kind, th * d_k + c);
    }
    for (int32_t r = 0; r < d_v; ++r) {
        vt[r] = oracle_load(v, kind, th * d_v + r);
        at[r] = (double)alpha[th * d_v + r];
    }
}

static void oracle_backward_pair(const void* q, const void* k, const void* v, int kind,
                                 const float* alpha, const float* beta, const double* S0,
                                 const double* dO, const double* dS_T,
                                 int64_t t_begin, int64_t t_end, int32_t n, int32_t h,
                                 int32_t H, int32_t d_k, int32_t d_v,
                                 double* dq, double* dk, double* dv, double* dalpha,
                                 double* dbeta, double* dS0, oracle_bwd_scratch* w)
{
    const int64_t sz = (int64_t)d_v * d_k;
    const int64_t state_off = ((int64_t)n * H + h) * sz;
    const int64_t L = t_end - t_begin;
    const int64_t nseg = (L + OR_SEG - 1) / OR_SEG;
    /* tape[0 .. nseg]: states at segment starts; tape[nseg + 1 + j]: state after
     * token j of the segment being differentiated (j = 0 .. OR_SEG - 1) */
    double* kept = w->tape;
    double* seg = w->tape + (nseg + 1) * sz;

    if (S0) memcpy(kept, S0 + state_off, sizeof(double) * (size_t)sz);
    else memset(kept, 0, sizeof(double) * (size_t)sz);
    for (int64_t s = 0; s < nseg; ++s) {
        const double* cur = kept + s * sz;
        double* nxt = kept + (s + 1) * sz;
        memcpy(nxt, cur, sizeof(double) * (size_t)sz);
        const int64_t a = t_begin + s * OR_SEG, e = a + OR_SEG < t_end ? a + OR_SEG : t_end;
        for (int64_t t = a; t < e; ++t) {
            const int64_t th = t * H + h;
            oracle_load_token(q, k, v, kind, alpha, th, d_k, d_v, w->qt, w->kt, w->vt, w->at);
            /* in place is safe: each row is read before it is written */
            oracle_step(nxt, nxt, w->kt, w->vt, w->at, (double)beta[th], d_k, d_v);
        }
    }

    /* D = dL/dS_T */
    if (dS_T) memcpy(w->D, dS_T + state_off, sizeof(double) * (size_t)sz);
    else memset(w->D, 0, sizeof(double) * (size_t)sz);

    for (int64_t s = nseg - 1; s >= 0; --s) {
        const int64_t a = t_begin + s * OR_SEG, e = a + OR_SEG < t_end ? a + OR_SEG : t_end;
        /* refill the states after each token of this segment */
        for (int64_t t = a; t < e; ++t) {
            const int64_t th = t * H + h;
            oracle_load_token(q, k, v, kind, alpha, th, d_k, d_v, w->qt, w->kt, w->vt, w->at);
            const double* prev = t == a ? kept + s * sz : seg + (t - a - 1) * sz;
            oracle_step(prev, seg + (t - a) * sz, w->kt, w->vt, w->at, (double)beta[th], d_k, d_v);
        }
        for (int64_t t = e - 1; t >= a; --t) {
            const int64_t th = t * H + h;
            oracle_load_token(q, k, v, kind, alpha, th, d_k, d_v, w->qt, w->kt, w->vt, w->at);
            const double b = (double)(beta[th]);
            const double* S_t = seg + (t - a) * sz;
            const double* S_prev = t == a ? kept + s * sz : seg + (t - a - 1) * sz;
            for (int32_t r = 0; r < d_v; ++r) w->dot[r] = dO[th * d_v + r];

            /* output: D += do q^T, dq = S_t^T do */
            for (int32_t r = 0; r < d_v; ++r) {
                double* Dr = w->D + (int64_t)r * d_k;
                for (int32_t c = 0; c < d_k; ++c) Dr[c] += w->dot[r] * w->qt[c];
            }
            for (int32_t c = 0; c < d_k; ++c) {
                double acc = 0.0;
                for (int32_t r = 0; r < d_v; ++r) acc += S_t[(int64_t)r * d_k + c] * w->dot[r];
                dq[th * d_k + c] = acc;
            }
            /* forget gating and predict again: S~ and u = v - S~ k */
            for (int32_t r = 0; r < d_v; ++r) {
                const double* src = S_prev + (int64_t)r * d_k;
                double* row = w->Stl + (int64_t)r * d_k;
                double pred = 0.0;
                for (int32_t c = 0; c < d_k; ++c) {
                    row[c] = w->at[r] * src[c];
                    pred += row[c] * w->kt[c];
                }
                w->u[r] = w->vt[r] - pred;
            }
            /* memory updating: g = D k, dv, dbeta, dk */
            double db = 0.0;
            for (int32_t r = 0; r < d_v; ++r) {
                const double* Dr = w->D + (int64_t)r * d_k;
                double acc = 0.0;
                for (int32_t c = 0; c < d_k; ++c) acc += Dr[c] * w->kt[c];
                w->g[r] = acc;
                dv[th * d_v + r] = b * acc;
                db += w->u[r] * acc;
            }
            dbeta[th] = db;
            for (int32_t c = 0; c < d_k; ++c) {
                double du = 0.0, sg = 0.0;
                for (int32_t r = 0; r < d_v; ++r) {
                    du += w->D[(int64_t)r * d_k + c] * w->u[r];
                    sg += w->Stl[(int64_t)r * d_k + c] * w->g[r];
                }
                dk[th * d_k + c] = b * (du - sg);
            }
            /* dS~ = D - beta g k^T; dalpha = rowwise <dS~, S_{t-1}>; D = diag(alpha) dS~ */
            for (int32_t r = 0; r < d_v; ++r) {
                double* Dr = w->D + (int64_t)r * d_k;
                const double* Pr = S_prev + (int64_t)r * d_k;
                double da = 0.0;
                for (int32_t c = 0; c < d_k; ++c) {
                    Dr[c] = Dr[c] - b * w->g[r] * w->kt[c];
                    da += Dr[c] * Pr[c];
                }
                dalpha[th * d_v + r] = da;
                for (int32_t c = 0; c < d_k; ++c) Dr[c] = w->at[r] * Dr[c];
            }
        }
    }
    if (dS0) memcpy(dS0 + state_off, w->D, sizeof(double) * (size_t)sz);
}

/*
 * Gradients of L = sum(dO * o) + sum(dS_T * S_T) for the packed batch that
 * kda_oracle_prefill runs (same input layouts and checks, same return codes).
 *   dO    [T_total][H][d_v] fp64          dS_T  [N][H][d_v][d_k] fp64 or NULL (zeros)
 *   dq,dk [T_total][H][d_k] fp64 out      dv, dalpha [T_total][H][d_v] fp64 out
 *   dbeta [T_total][H] fp64 out           dS0   [N][H][d_v][d_k] fp64 out or NULL
 * Tokens past cu_seqlens[num_seqs] get zero gradients.
 */
int kda_oracle_backward(const void* q, const void* k, const void* v, int kind,
                        const float* alpha, const float* beta, const double* S0,
                        const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                        int32_t H, int32_t d_k, int32_t d_v,
                        const double* dO, const double* dS_T,
                        double* dq, double* dk, double* dv, double* dalpha, double* dbeta,
                        double* dS0, int32_t nthreads)
{
    if (num_seqs < 0 || H <= 0 || d_k <= 0 || d_v <= 0 || (kind != 0 && kind != 1)) return 1;
    if (!cu_seqlens || (num_seqs > 0 && (!q || !k || !v || !alpha || !beta || !dO || !dq ||
                                         !dk || !dv || !dalpha || !dbeta))) return 1;
    if (cu_seqlens[0] != 0) return 2;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 2;
    if ((int64_t)cu_seqlens[num_seqs] > total_tokens) return 2;
    if (num_seqs == 0) return 0;

    memset(dq, 0, sizeof(double) * (size_t)total_tokens * H * d_k);
    memset(dk, 0, sizeof(double) * (size_t)total_tokens * H * d_k);
    memset(dv, 0, sizeof(double) * (size_t)total_tokens * H * d_v);
    memset(dalpha, 0, sizeof(double) * (size_t)total_tokens * H * d_v);
    memset(dbeta, 0, sizeof(double) * (size_t)total_tokens * H);

    int64_t max_len = 0;
    for (int32_t n = 0; n < num_seqs; ++n) {
        const int64_t len = (int64_t)cu_seqlens[n + 1] - cu_seqlens[n];
        if (len > max_len) max_len = len;
    }
    const int64_t sz = (int64_t)d_v * d_k;
    const int64_t tape_states = (max_len + OR_SEG - 1) / OR_SEG + 1 + OR_SEG;
    const int64_t pairs = (int64_t)num_seqs * H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(|: failed)
#endif
    {
        oracle_bwd_scratch w;
        w.tape = (double*)malloc(sizeof(double) * (size_t)(tape_states * sz));
        w.D = (double*)malloc(sizeof(double) * (size_t)sz);
        w.Stl = (double*)malloc(sizeof(double) * (size_t)sz);
        w.kt = (double*)malloc(sizeof(double) * (size_t)d_k);
        w.qt = (double*)malloc(sizeof(double) * (size_t)d_k);
        w.vt = (double*)malloc(sizeof(double) * (size_t)d_v);
        w.at = (double*)malloc(sizeof(double) * (size_t)d_v);
        w.dot = (double*)malloc(sizeof(double) * (size_t)d_v);
        w.g = (double*)malloc(sizeof(double) * (size_t)d_v);
        w.u = (double*)malloc(sizeof(double) * (size_t)d_v);
        const int have = w.tape && w.D && w.Stl && w.kt && w.qt && w.vt && w.at && w.dot &&
                         w.g && w.u;
        if (!have) failed = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t p = 0; p < pairs; ++p) {
            if (!have) continue;
            const int32_t n = (int32_t)(p / H), h = (int32_t)(p % H);
            oracle_backward_pair(q, k, v, kind, alpha, beta, S0, dO, dS_T, cu_seqlens[n],
                                 cu_seqlens[n + 1], n, h, H, d_k, d_v, dq, dk, dv, dalpha,
                                 dbeta, dS0, &w);
        }
        free(w.tape); free(w.D); free(w.Stl); free(w.kt); free(w.qt); free(w.vt);
        free(w.at); free(w.dot); free(w.g); free(w.u);
    }
    return failed ? 3 : 0;
}

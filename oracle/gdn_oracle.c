/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet prompt-prefill
 * path (conv -> SiLU -> L2 norm -> gates -> gated delta-rule scan -> gated
 * RMSNorm).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * Everything is computed in IEEE double, token by token, in the order the
 * method defines it, with no blocking, fusion or reordering.  All arrays are
 * dense row-major; callers widen fp16/fp32 inputs to double exactly.
 *
 * Sources (the pages benchmark these stages but never print the equations;
 * the stage definitions below follow the method statement the stages are
 * built to, and each function names the page passage it is consistent with):
 *   - "Round 30 Track C Audit: gdn_pre, gdn_post, and gdn_scanr_4", section 1
 *     (gdn_pre: 4-tap conv loop, history written at the last token, per-head
 *     q/k sum-of-squares reductions; gdn_post: per-head sum-of-squares
 *     reduction, f32/fp16 output switch).
 *   - "round 10 track b: gdn vectorization and scan", source and execution
 *     (hk=16, hv=48, channels=10240, eps=1e-6) and variants (each conv
 *     output is four multiply-adds taken in tap order; the history buffer is
 *     laid out channel by channel; SiLU on every channel).
 *   - "opus_r25_gdn -- round 25 track A", shipped (gdn_post sigmoid gate,
 *     gamma) and the scan's per-token loop (state decay, k/q reductions).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* ---- scalar activations (plain definitions) ---------------------------- */

/* logistic sigmoid 1/(1+e^-x), evaluated without overflow for either sign */
double gdn_oracle_sigmoid(double x)
{
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

/* SiLU(x) = x * sigmoid(x) */
double gdn_oracle_silu_scalar(double x) { return x * gdn_oracle_sigmoid(x); }

/* softplus(x) = log(1 + e^x), written as max(x,0) + log1p(e^-|x|) so that it
 * is exact for every finite x (no cut-over threshold). */
double gdn_oracle_softplus(double x)
{
    double m = x > 0.0 ? x : 0.0;
    return m + log1p(exp(-fabs(x)));
}

/* ---- stage 1a: width-4 causal depthwise conv with carried history ------ */
/*
 * y[t][c] = sum_{m=0..3} w[c][m] * xt(t-3+m, c), where xt(s,c) = x[s][c] for
 * s >= 0 and hist[c][3+s] for s in {-3,-2,-1} (hist[c][0] is the oldest).
 * Tap m=3 multiplies the current token.  No bias.  The history left for the
 * next call is the last three inputs: hist_out[c][i] = xt(T-3+i, c); when
 * T < 3 part of it comes from the old history.
 * (Round 30 audit section 1: the unrolled m = 0..3 conv loop and the
 * t == T-1 history write; round 10 variants: four multiply-adds per output
 * in tap order, history laid out channel by channel.)
 */
static double conv_tap(int64_t s, int64_t c, int64_t C, const double* x, const double* hist)
{
    return s >= 0 ? x[s * C + c] : hist[c * 3 + (3 + s)];
}

void gdn_oracle_conv(int64_t T, int64_t C, const double* x, const double* w,
                     const double* hist, double* y, double* hist_out)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int m = 0; m < 4; ++m)
                acc += w[c * 4 + m] * conv_tap(t - 3 + m, c, C, x, hist);
            y[t * C + c] = acc;
        }
    if (hist_out)
        for (int64_t c = 0; c < C; ++c)
            for (int i = 0; i < 3; ++i)
                hist_out[c * 3 + i] = conv_tap(T - 3 + i, c, C, x, hist);
}

/* ---- stage 1b: SiLU on every channel ------------------------------------ */
void gdn_oracle_silu(int64_t n, const double* in, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = gdn_oracle_silu_scalar(in[i]);
}

/* ---- stage 1c: per-head L2 normalisation --------------------------------- */
/* out = in / sqrt(sum(in^2) + eps) for each row of length d (one q or k head).
 * (Round 30 audit section 1: the per-key-head sum-of-squares reductions
 * sq/sk; eps = 1e-6 from the round 10 source-and-execution list.) */
void gdn_oracle_l2norm(int64_t rows, int64_t d, double eps, const double* in, double* out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double* x = in + r * d;
        double ss = 0.0;
        for (int64_t i = 0; i < d; ++i) ss += x[i] * x[i];
        double inv = 1.0 / sqrt(ss + eps);
        for (int64_t i = 0; i < d; ++i) out[r * d + i] = x[i] * inv;
    }
}

/* ---- stage 1d: decay and write-strength gates ---------------------------- */
/* lam = -exp(A_log[h]) * softplus(a[t][h] + dt_bias[h]);  g = exp(lam);
 * beta = sigmoid(b[t][h]).  (The scan's per-token (g, beta) pair, read
 * through the gb buffer with a stride of hv per token, round 30 audit
 * section 1.) */
void gdn_oracle_gates(int64_t T, int64_t hv, const double* a, const double* b,
                      const double* A_log, const double* dt_bias,
                      double* g, double* lam, double* beta)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < hv; ++h) {
            double l = -exp(A_log[h]) * gdn_oracle_softplus(a[t * hv + h] + dt_bias[h]);
            if (lam) lam[t * hv + h] = l;
            if (g) g[t * hv + h] = exp(l);
            if (beta) beta[t * hv + h] = gdn_oracle_sigmoid(b[t * hv + h]);
        }
}

/* ---- stage 2: gated delta-rule recurrence, one value head ----------------- */
/*
 * State S in R^{dk x dv} (S[i][j], i over keys, j over values), per token t:
 *     S <- g_t * S
 *     u  = beta_t * (v_t - S^T k_t)
 *     S <- S + k_t u^T
 *     o_t = S^T (q_t / sqrt(dk))
 * q, k, v, g, beta are read with the given strides (elements between
 * consecutive tokens).  S0 and S_out are [dk][dv].  S_out may equal S0.
 * (Round 30 audit section 1: gdn_scan_r's per-token loop keeps the fp32
 * state in registers, decays and updates it and forms the k and q dot
 * products against it; this is that recurrence, written plainly in fp64.)
 */
void gdn_oracle_scan_head(int64_t T, int64_t dk, int64_t dv,
                          const double* q, int64_t q_stride,
                          const double* k, int64_t k_stride,
                          const double* v, int64_t v_stride,
                          const double* g, const double* beta, int64_t gb_stride,
                          const double* S0, double* o, int64_t o_stride,
                          double* S_out)
{
    const double qscale = 1.0 / sqrt((double)dk);
    /* S plus two length-dv accumulators.  Each dot product over i is still
     * summed in increasing i; the j loop is innermost only so that the row
     * S[i][*] is walked contiguously. */
    double* S = (double*)malloc(sizeof(double) * (size_t)(dk * dv + 2 * dv));
    double* sk = S + dk * dv;
    double* u = sk + dv;
    for (int64_t i = 0; i < dk * dv; ++i) S[i] = S0[i];
    for (int64_t t = 0; t < T; ++t) {
        const double* qt = q + t * q_stride;
        const double* kt = k + t * k_stride;
        const double* vt = v + t * v_stride;
        const double gt = g[t * gb_stride];
        const double bt = beta[t * gb_stride];
        for (int64_t i = 0; i < dk * dv; ++i) S[i] *= gt;            /* S <- g S      */
        for (int64_t j = 0; j < dv; ++j) sk[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)                              /* sk = S^T k    */
            for (int64_t j = 0; j < dv; ++j) sk[j] += S[i * dv + j] * kt[i];
        for (int64_t j = 0; j < dv; ++j) u[j] = bt * (vt[j] - sk[j]); /* u = b(v-S^Tk) */
        for (int64_t i = 0; i < dk; ++i)                              /* S += k u^T    */
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * u[j];
        double* ot = o + t * o_stride;                                /* o = S^T q/sqrt(dk) */
        for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i) {
            const double qi = qt[i] * qscale;
            for (int64_t j = 0; j < dv; ++j) ot[j] += S[i * dv + j] * qi;
        }
    }
    for (int64_t i = 0; i < dk * dv; ++i) S_out[i] = S[i];
    free(S);
}

/*
 * All (or a subset of) value heads of one sequence.  Layouts:
 *   q, k [T][hk][dk]; v, o [T][hv][dv]; g, beta [T][hv]; S0, S_out [hv][dk][dv].
 * Value head h reads key head h / (hv/hk).  heads == NULL means every head;
 * otherwise only the n_heads listed heads are computed (outputs of the other
 * heads are left untouched).  Heads run in parallel when built with OpenMP.
 */
#ifdef _OPENMP
#include <omp.h>
#endif
int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void gdn_oracle_scan(int64_t T, int64_t hk, int64_t hv, int64_t dk, int64_t dv,
                     const double* q, const double* k, const double* v,
                     const double* g, const double* beta, const double* S0,
                     const int32_t* heads, int64_t n_heads,
                     double* o, double* S_out)
{
    const int64_t group = hv / hk;
    const int64_t n = heads ? n_heads : hv;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t idx = 0; idx < n; ++idx) {
        const int64_t h = heads ? heads[idx] : idx;
        const int64_t j = h / group;
        gdn_oracle_scan_head(T, dk, dv,
                             q + j * dk, hk * dk,
                             k + j * dk, hk * dk,
                             v + h * dv, hv * dv,
                             g + h, beta + h, hv,
                             S0 + h * dk * dv,
                             o + h * dv, hv * dv,
                             S_out + h * dk * dv);
    }
}

/* ---- stage 3: gated RMSNorm ---------------------------------------------- */
/* y = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z), per row of dv values
 * (one (token, value head) pair); gamma has dv entries shared by all heads.
 * (Round 30 audit section 1 and round 25 "shipped": gdn_post's per-head
 * sum-of-squares reduction, gamma load and sigmoid gate.) */
void gdn_oracle_post(int64_t rows, int64_t dv, double eps, const double* o,
                     const double* z, const double* gamma, double* y)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double* orow = o + r * dv;
        const double* zrow = z + r * dv;
        double ss = 0.0;
        for (int64_t i = 0; i < dv; ++i) ss += orow[i] * orow[i];
        double inv = 1.0 / sqrt(ss / (double)dv + eps);
        for (int64_t i = 0; i < dv; ++i)
            y[r * dv + i] = orow[i] * inv * gamma[i] * gdn_oracle_silu_scalar(zrow[i]);
    }
}

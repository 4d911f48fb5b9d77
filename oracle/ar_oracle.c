/*
 * ar_oracle.c -- plain CPU fp64 oracle for the fused decode-layer boundary
 * (MoE finalize + shared-expert add + TP all-reduce arithmetic + residual
 * add + RMSNorm).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and the CPU-baseline
 * leg of bench.py use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (the plain definition; each loop below is one sum of it).
 * For token t and column j, all arithmetic in IEEE binary64:
 *
 *   y[t,j]   = sum_{r<R} ( sum_{k<K} w[t,k] * E_r[perm[t*K+k], j] + S_r[t,j] )
 *   h[t,j]   = y[t,j] + residual[t,j]                        -> residual_out
 *   ms[t]    = (1/H) * sum_j h[t,j]^2
 *   out[t,j] = h[t,j] / sqrt(ms[t] + eps) * (gamma[j] + weight_bias)
 *
 * Sources:
 *  - sglang PR #37196 "[Comm] Share the CuTe DSL AR fusion core and wire it
 *    for DeepSeek-V3 / GLM-5.x", Motivation: the fused op folds the MoE
 *    finalize, the shared-expert add and the post-experts all-reduce into the
 *    next layer's input RMSNorm.
 *  - same page, Modifications section 1: the norm scales by
 *    (gamma + weight_bias); Gemma-style weights already hold checkpoint + 1,
 *    so both norm flavours use weight_bias = 0.
 *  - same page, Modifications section 2: the DeepSeek-V3 shared expert has no
 *    sigmoid gate (it is added unmodified), and a replicated shared expert
 *    must not be folded in: S_r is a per-rank partial, summed once over r.
 *    The Qwen-style shared expert does carry a per-token sigmoid gate, applied
 *    to the shared output before the fused add: with gate logits g[t] the
 *    shared term becomes sigmoid(g[t]) * S_r[t,j] (oracle_..._gated).
 *  - sglang PR #37104 "perf(mtp): fuse trailing TP all-reduce with final
 *    RMSNorm", Changes: a residual is mandatory.
 *
 * Every product w*E is exact in binary64 (24 + 8 significand bits <= 53), so
 * the only roundings are the running sum of at most R*(K+1)+1 terms and the
 * final sqrt/divide.  Build with -ffp-contract=off so no fused multiply-add
 * changes the rounding between machines.
 *
 * bf16 values arrive as raw uint16 bit patterns and are decoded by placing
 * them in the top half of an IEEE binary32 word.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_PERM_RANGE (-2)

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a binary64 value to the nearest bfloat16 value (ties to even), in one
 * step (no detour through binary32, so no double rounding).  bfloat16 has 8
 * significant bits, exponent range of binary32: smallest normal 2^-126,
 * smallest subnormal 2^-133, largest finite (2 - 2^-7) * 2^127. */
double oracle_round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int e;
    (void)frexp(x, &e);            /* x = m * 2^e with 0.5 <= |m| < 1 */
    int q = e - 8;                 /* weight of the 8th significant bit */
    if (q < -133)
        q = -133;                  /* subnormal range: fixed quantum */
    double r = nearbyint(ldexp(x, -q));   /* default mode: ties to even */
    double y = ldexp(r, q);
    const double bf16_max = ldexp(255.0, 120);   /* (2 - 2^-7) * 2^127 */
    if (fabs(y) > bf16_max)
        y = copysign(INFINITY, x);
    return y;
}

void oracle_round_bf16_array(const double *x, double *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = oracle_round_bf16(x[i]);
}

/* y and h of one token row (steps: routed gather-sum, shared add, rank sum,
 * residual add).  abs_row, when non-NULL, receives sum |term| per column:
 * the scale of the cancellation the sum can suffer. */
static void oracle_row_sum(int64_t t, int R, int K, int H,
                           const uint16_t *const *E, const int32_t *perm,
                           const float *w, const uint16_t *const *S,
                           const float *gate, const uint16_t *residual,
                           double *h_row, double *abs_row)
{
    /* shared-expert gate of this token: sigmoid of its logit (1 if none) */
    const double g = gate ? 1.0 / (1.0 + exp(-(double)gate[t])) : 1.0;
    for (int j = 0; j < H; ++j) {
        double y = 0.0, a = 0.0;
        for (int r = 0; r < R; ++r) {
            double y_r = 0.0;                    /* rank r's partial */
            for (int k = 0; k < K; ++k) {
                int64_t row = perm[t * K + k];
                double term = (double)w[t * K + k] *
                              bf16_bits_to_double(E[r][row * H + j]);
                y_r += term;
                a += fabs(term);
            }
            if (S) {
                double s = g * bf16_bits_to_double(S[r][t * H + j]);
                y_r += s;
                a += fabs(s);
            }
            y += y_r;                            /* the all-reduce sum */
        }
        double res = bf16_bits_to_double(residual[t * H + j]);
        h_row[j] = y + res;
        if (abs_row)
            abs_row[j] = a + fabs(res);
    }
}

/* RMSNorm of one row: out = h / sqrt(mean(h^2) + eps) * (gamma + weight_bias).
 * With h_bf16 set the norm reads h rounded to bf16 (the alternative reading
 * in which the norm consumes the stored bf16 residual_out). */
static void oracle_row_norm(int H, const double *h_row, const uint16_t *gamma,
                            double weight_bias, double eps, int h_bf16,
                            double *out_row)
{
    double ssq = 0.0;
    for (int j = 0; j < H; ++j) {
        double hj = h_bf16 ? oracle_round_bf16(h_row[j]) : h_row[j];
        ssq += hj * hj;
    }
    double ms = ssq / (double)H;
    double denom = sqrt(ms + eps);
    for (int j = 0; j < H; ++j) {
        double hj = h_bf16 ? oracle_round_bf16(h_row[j]) : h_row[j];
        double g = bf16_bits_to_double(gamma[j]) + weight_bias;
        out_row[j] = hj / denom * g;
    }
}

/*
 * Full operator.  Shapes (row-major):
 *   E[r]      bf16 bits [rows_e, H] for r < R        (unused when K == 0)
 *   perm      int32 [T, K]  gather index into E rows  (unused when K == 0)
 *   w         fp32  [T, K]                             (unused when K == 0)
 *   S[r]      bf16 bits [T, H], or S == NULL (no shared term)
 *   residual  bf16 bits [T, H]   (required)
 *   gamma     bf16 bits [H]
 * Outputs (binary64, unrounded):
 *   h_out     [T, H]  residual_out before storage rounding
 *   out       [T, H]  normalised output before storage rounding
 *   abs_terms [T, H]  sum of |terms| of h (may be NULL)
 * Returns ORACLE_OK, ORACLE_BAD_ARG, or ORACLE_PERM_RANGE when some perm value
 * is outside [0, rows_e) (nothing is computed then).
 */
static int oracle_run(int R, int K, int H, int64_t T, int64_t rows_e,
                      const uint16_t *const *E, const int32_t *perm, const float *w,
                      const uint16_t *const *S, const float *gate,
                      const uint16_t *residual, const uint16_t *gamma,
                      double weight_bias, double eps, int h_bf16, double *h_out,
                      double *out, double *abs_terms)
{
    if (R < 1 || K < 0 || H < 1 || T < 0 || !residual || !gamma || !h_out ||
        !out)
        return ORACLE_BAD_ARG;
    if (K > 0 && (!E || !perm || !w || rows_e < 1))
        return ORACLE_BAD_ARG;
    if (K == 0 && !S)
        return ORACLE_BAD_ARG;   /* nothing to reduce */
    if (gate && !S)
        return ORACLE_BAD_ARG;   /* a gate needs a shared term */
    for (int64_t i = 0; i < T * (int64_t)K; ++i)
        if (perm[i] < 0 || (int64_t)perm[i] >= rows_e)
            return ORACLE_PERM_RANGE;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double *h_row = h_out + t * H;
        oracle_row_sum(t, R, K, H, E, perm, w, S, gate, residual, h_row,
                       abs_terms ? abs_terms + t * H : NULL);
        oracle_row_norm(H, h_row, gamma, weight_bias, eps, h_bf16,
                        out + t * H);
    }
    return ORACLE_OK;
}

int oracle_ar_finalize_rmsnorm(int R, int K, int H, int64_t T, int64_t rows_e,
                               const uint16_t *const *E, const int32_t *perm,
                               const float *w, const uint16_t *const *S,
                               const uint16_t *residual, const uint16_t *gamma,
                               double weight_bias, double eps, int h_bf16,
                               double *h_out, double *out, double *abs_terms)
{
    return oracle_run(R, K, H, T, rows_e, E, perm, w, S, NULL, residual, gamma,
                      weight_bias, eps, h_bf16, h_out, out, abs_terms);
}

/* The same with the Qwen-style per-token sigmoid gate on the shared term:
 * gate[t] is the fp32 gate logit of token t (required, as is S). */
int oracle_ar_finalize_rmsnorm_gated(int R, int K, int H, int64_t T,
                                     int64_t rows_e, const uint16_t *const *E,
                                     const int32_t *perm, const float *w,
                                     const uint16_t *const *S, const float *gate,
                                     const uint16_t *residual,
                                     const uint16_t *gamma, double weight_bias,
                                     double eps, int h_bf16, double *h_out,
                                     double *out, double *abs_terms)
{
    if (!gate || !S)
        return ORACLE_BAD_ARG;
    return oracle_run(R, K, H, T, rows_e, E, perm, w, S, gate, residual, gamma,
                      weight_bias, eps, h_bf16, h_out, out, abs_terms);
}

/* Trailing all-reduce + residual RMSNorm without a MoE term: the K = 0 case,
 * with the R partials in place of S (sglang PR #37104, Changes). */
int oracle_ar_rmsnorm(int R, int H, int64_t T, const uint16_t *const *partials,
                      const uint16_t *residual, const uint16_t *gamma,
                      double weight_bias, double eps, int h_bf16,
                      double *h_out, double *out, double *abs_terms)
{
    if (!partials)
        return ORACLE_BAD_ARG;
    return oracle_ar_finalize_rmsnorm(R, 0, H, T, 0, NULL, NULL, NULL,
                                      partials, residual, gamma, weight_bias,
                                      eps, h_bf16, h_out, out, abs_terms);
}

/*
 * All-reduce + mHC residual write-back ("hc_post").  sglang PR #42020 (ROCm
 * aiter fused all-reduce + mHC hc_post for GLM-5.3-Flash), Summary and Scope:
 * an mHC layer writes its FFN output back as two launches -- the FFN's
 * tensor-parallel all-reduce, then hc_post, which reads the reduced output
 * back and mixes it into the hc_mult = 4 residual streams -- and the fused
 * kernel does both in one pass (at most 16 tokens in serving).
 *
 * The page gives no formula for the mix.  Reading taken here, the plainest
 * one the page supports (a per-token linear mix of the reduced output and the
 * incoming streams, as in hyper-connection write-backs):
 *
 *   y[t,j]     = sum_{r<R} P_r[t,j]                          (the all-reduce)
 *   out[t,i,j] = post[t,i] * y[t,j] + sum_{k<hc} comb[t,i,k] * x[t,k,j]
 *
 * P_r bf16 [T, H]; x (incoming streams) bf16 [T, hc, H]; post fp32 [T, hc];
 * comb fp32 [T, hc, hc] (row i mixes the streams into output stream i).
 * PARITY UNPINNED against the pages (they do not define hc_post): the tests
 * pin this code to the reading above only.  Every product is exact in
 * binary64; the only roundings are the sums.
 */
int oracle_ar_mhc_post(int R, int H, int hc, int64_t T,
                       const uint16_t *const *partials, const uint16_t *x,
                       const float *post, const float *comb, double *out)
{
    if (R < 1 || H < 1 || hc < 1 || T < 0 || !partials || !x || !post ||
        !comb || !out)
        return ORACLE_BAD_ARG;
    for (int r = 0; r < R; ++r)
        if (!partials[r])
            return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < H; ++j) {
            double y = 0.0;
            for (int r = 0; r < R; ++r)
                y += bf16_bits_to_double(partials[r][t * H + j]);
            for (int i = 0; i < hc; ++i) {
                double o = (double)post[t * hc + i] * y;
                for (int k = 0; k < hc; ++k)
                    o += (double)comb[(t * hc + i) * hc + k] *
                         bf16_bits_to_double(x[(t * hc + k) * H + j]);
                out[(t * hc + i) * H + j] = o;
            }
        }
    }
    return ORACLE_OK;
}

/* Thread control for the timed CPU baseline (OpenMP over token rows). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

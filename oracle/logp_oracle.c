/*
 * FP64 CPU oracle for the selected-token log-probability and its gradient.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product path
 * never does, and it shares no code, header or constant with the CUDA
 * library.
 *
 * What it follows (RL-Kernel pages):
 *   - issue #241 "TP-aware deterministic logprob", Background + Goal: the
 *     selected-token logprob is the target logit minus the log-sum-exp over
 *     the vocabulary; PR 3 bullets: per-shard (max, sumexp) partials and the
 *     merge M = max m_l, S = sum s_l exp(m_l - M), LSE = M + log S.
 *   - PR #495 "zero-workspace fused backward", Summary item 2: the gradient
 *     is grad * (one_hot - softmax); Behavior changes: a target outside
 *     [0, V) (for example the ignore index -100) gives logp 0 and an exactly
 *     zero gradient row.
 *   - PR #314 "Deterministic config option", ReductionSpec text: padded
 *     columns count as -inf, and (-inf, 0) is the identity partial.
 *
 * Everything is computed in IEEE double from the exact inputs with a plain
 * two-pass log-sum-exp.  Compile with -ffp-contract=off so that x86 and Arm
 * hosts round identically.
 *
 * Variants (the same definitions, generalised):
 *   - logits in BF16, FP16 or FP32 (PR #495 Tests: accuracy for
 *     FP32/BF16/FP16 against an FP64 reference), widened exactly;
 *   - a temperature: the logits are scaled by s = 1/T before the log-softmax
 *     (PR #495, the provider experiment: rollout logprobs at temperature 1.0
 *     and 0.7), so LSE = log sum exp(s x), logp = s x_y - LSE and, by the chain
 *     rule, d = s g (onehot - exp(s x - LSE));
 *   - an explicit active-row mask (PR #314, MaskMode explicit_active_mask):
 *     a row is active only if its mask byte is nonzero;
 *   - the fused LM head (linear_logp): the logits are formed from hidden
 *     states and weight rows first (oracle_linear_logp).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- BF16 <-> double --------------------------------------------------- */

/* A BF16 value is the top 16 bits of an IEEE binary32; widen it exactly. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double straight to the nearest BF16 (ties to even), without an
 * intermediate binary32 rounding (which could round twice).  BF16 has an
 * 8-bit significand and binary32's exponent range, so the spacing of BF16
 * values in [2^e, 2^(e+1)) is 2^(e-7), and below 2^-126 it is 2^-133. */
uint16_t oracle_round_bf16(double d) {
    if (isnan(d)) return 0x7fc0;
    int neg = signbit(d) ? 1 : 0;
    uint16_t sign = neg ? 0x8000 : 0;
    double a = fabs(d);
    if (isinf(a)) return sign | 0x7f80;
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);              /* a = f * 2^e with f in [0.5, 1) */
    int q = (e - 1) - 7;             /* exponent of one BF16 unit in the last place */
    if (q < -133) q = -133;          /* subnormal BF16 spacing */
    double r = nearbyint(ldexp(a, -q));  /* default mode: nearest, ties to even */
    double val = ldexp(r, q);
    /* largest finite BF16 is (2 - 2^-7) * 2^127 */
    if (val > ldexp(255.0, 120)) return sign | 0x7f80;
    float f = (float)val;            /* exact: val is a BF16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7fff));
}

void oracle_round_bf16_array(const double* in, uint16_t* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_round_bf16(in[i]);
}

void oracle_bf16_to_double_array(const uint16_t* in, double* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = bf16_bits_to_double(in[i]);
}

/* ---- FP16 and element access by dtype ------------------------------------- */

enum { DT_BF16 = 0, DT_F16 = 1, DT_F32 = 2 };

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
 * subnormals below 2^-14 with spacing 2^-24. */
static double f16_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0x1f) v = f ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)f, -24);
    else v = ldexp((double)(f | 0x400), e - 25);
    return sign ? -v : v;
}

/* Round a double to the nearest binary16 (ties to even); overflow to inf at
 * 65520 = max + half an ulp. */
uint16_t oracle_round_f16(double d) {
    if (isnan(d)) return 0x7e00;
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    double a = fabs(d);
    if (isinf(a)) return sign | 0x7c00;
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);
    int q = (e - 1) - 10;            /* exponent of one unit in the last place */
    if (q < -24) q = -24;            /* subnormal spacing */
    double r = nearbyint(ldexp(a, -q));
    double val = ldexp(r, q);
    if (val >= 65520.0) return sign | 0x7c00;
    /* encode val (exactly representable) */
    if (val < ldexp(1.0, -14)) return sign | (uint16_t)ldexp(val, 24);
    int ev;
    double fr = frexp(val, &ev);     /* val = fr * 2^ev, fr in [0.5, 1) */
    uint16_t bits = (uint16_t)(((ev - 1 + 15) << 10) | ((uint16_t)ldexp(fr * 2.0 - 1.0, 10)));
    return sign | bits;
}

void oracle_round_f16_array(const double* in, uint16_t* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_round_f16(in[i]);
}

void oracle_f16_to_double_array(const uint16_t* in, double* out, int64_t count) {
    for (int64_t i = 0; i < count; ++i) out[i] = f16_bits_to_double(in[i]);
}

/* Element c of row t of an [n, ld] logit matrix of the given dtype, exactly. */
static double elem(const void* x, int dtype, int64_t ld, int64_t t, int64_t c) {
    int64_t i = t * ld + c;
    if (dtype == DT_F32) return (double)((const float*)x)[i];
    if (dtype == DT_F16) return f16_bits_to_double(((const uint16_t*)x)[i]);
    return bf16_bits_to_double(((const uint16_t*)x)[i]);
}

/* The value of the output dtype nearest to d (ties to even), as a double. */
static double round_to(double d, int dtype) {
    if (dtype == DT_F32) return (double)(float)d;  /* C conversion rounds to nearest even */
    if (dtype == DT_F16) return f16_bits_to_double(oracle_round_f16(d));
    return bf16_bits_to_double(oracle_round_bf16(d));
}

/* ---- row log-sum-exp ----------------------------------------------------- */

/* Plain two-pass log-sum-exp of the scaled row s * x over columns [c0, c1):
 * m = max s x, sum = sum exp(s x - m).  An all -inf range gives m = -inf and
 * sum = 0, the identity partial (PR #314, ReductionSpec). */
static void range_max_sumexp(const void* x, int dtype, int64_t ld, int64_t t, int64_t c0,
                             int64_t c1, double s, double* m_out, double* s_out) {
    double m = -INFINITY;
    for (int64_t c = c0; c < c1; ++c) {
        double v = s * elem(x, dtype, ld, t, c);
        if (v > m) m = v;
    }
    double acc = 0.0;
    if (m != -INFINITY) {
        for (int64_t c = c0; c < c1; ++c) {
            double v = s * elem(x, dtype, ld, t, c);
            if (v != -INFINITY) acc += exp(v - m);
        }
    }
    *m_out = m;
    *s_out = acc;
}

/* LSE = m + log(sum exp(s x - m)) over the whole row (-inf for an all -inf row). */
static double row_lse(const void* x, int dtype, int64_t ld, int64_t t, int64_t v, double s) {
    double m, acc;
    range_max_sumexp(x, dtype, ld, t, 0, v, s, &m, &acc);
    if (m == -INFINITY) return -INFINITY;
    return m + log(acc);
}

/* A row is active when its mask byte (if a mask is given) is nonzero and its
 * target names a real vocabulary column other than the ignore index (PR #495,
 * Behavior changes: out-of-range targets; PR #314 MaskMode). */
static int row_active(const int64_t* y, const uint8_t* mask, int64_t t, int64_t v,
                      int64_t ignore_index) {
    return (mask == 0 || mask[t] != 0) && y[t] >= 0 && y[t] < v && y[t] != ignore_index;
}

/* ---- vocab partials and their merge ---------------------------------------- */

/* Merge of k partials per row in index order (issue #241, PR 3 bullets):
 * M = max m_l, S = sum s_l exp(m_l - M), LSE = M + log S.  Identity
 * partials (m = -inf) contribute nothing; a row of identities has LSE -inf. */
void oracle_merge_partials(const double* pm, const double* ps, int64_t n,
                           int64_t k, double* lse) {
    for (int64_t t = 0; t < n; ++t) {
        const double* m = pm + t * k;
        const double* s = ps + t * k;
        double M = -INFINITY;
        for (int64_t j = 0; j < k; ++j)
            if (m[j] > M) M = m[j];
        if (M == -INFINITY) {
            lse[t] = -INFINITY;
            continue;
        }
        double S = 0.0;
        for (int64_t j = 0; j < k; ++j)
            if (m[j] != -INFINITY) S += s[j] * exp(m[j] - M);
        lse[t] = M + log(S);
    }
}

/* ---- entry points (dtype, scale s = 1/T, active mask) ----------------------- */

/* logp[t] = s x[t, y_t] - LSE_t for active rows (else 0), lse[t] = LSE_t,
 * LSE_t = log sum_v exp(s x[t, v]). */
void oracle_forward(const void* x, int dtype, int64_t n, int64_t v, int64_t ld,
                       const int64_t* y, int64_t ignore_index, const uint8_t* mask, double s,
                       double* logp, double* lse) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        double l = row_lse(x, dtype, ld, t, v, s);
        lse[t] = l;
        logp[t] = row_active(y, mask, t, v, ignore_index) ? s * elem(x, dtype, ld, t, y[t]) - l : 0.0;
    }
}

/* Dense gradient with respect to the unscaled logits:
 * d = s g (onehot - exp(s x - LSE)), the target column as -s g expm1(s x_y - LSE). */
void oracle_backward(const void* x, int dtype, int64_t n, int64_t v, int64_t ld,
                        const int64_t* y, int64_t ignore_index, const uint8_t* mask, double s,
                        const float* g, double* d, int64_t ld_d) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        double* dr = d + t * ld_d;
        if (!row_active(y, mask, t, v, ignore_index)) {
            for (int64_t c = 0; c < v; ++c) dr[c] = 0.0;
            continue;
        }
        double l = row_lse(x, dtype, ld, t, v, s);
        double gs = s * (double)g[t];
        for (int64_t c = 0; c < v; ++c) {
            double u = s * elem(x, dtype, ld, t, c) - l;
            dr[c] = (c == y[t]) ? -gs * expm1(u) : -gs * exp(u);
        }
    }
}

/* Streaming comparison of a gradient buffer dl[n, ld_out] in dtype out_dtype
 * with the FP64 gradient, one row at a time, never holding an FP64 [n, v]
 * array.  stats (doubles): [0] max |dl - d64|, [1] max |d64|,
 * [2] max |round(d64) - d64| (the error a correctly rounded result has);
 * counts (int64): [0] elements compared, [1] elements whose value differs from
 * the nearest out_dtype value of d64, [2] non-finite outputs where d64 is
 * finite.  Values are compared as numbers (+0 equals -0). */
void oracle_backward_compare(const void* x, int dtype, int64_t n, int64_t v, int64_t ld,
                                const int64_t* y, int64_t ignore_index, const uint8_t* mask,
                                double s, const float* g, const void* dl, int out_dtype,
                                int64_t ld_out, double* stats, int64_t* counts) {
    double max_diff = 0.0, max_d = 0.0, max_gap = 0.0;
    int64_t n_cmp = 0, n_bad = 0, n_nonfinite = 0;
#pragma omp parallel
    {
        double l_diff = 0.0, l_d = 0.0, l_gap = 0.0;
        int64_t l_cmp = 0, l_bad = 0, l_nf = 0;
#pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            int act = row_active(y, mask, t, v, ignore_index);
            double l = act ? row_lse(x, dtype, ld, t, v, s) : 0.0;
            double gs = s * (double)g[t];
            for (int64_t c = 0; c < v; ++c) {
                double d64 = 0.0;
                if (act) {
                    double u = s * elem(x, dtype, ld, t, c) - l;
                    d64 = (c == y[t]) ? -gs * expm1(u) : -gs * exp(u);
                }
                double crv = round_to(d64, out_dtype);
                double got = elem(dl, out_dtype, ld_out, t, c);
                double diff = fabs(got - d64);
                if (!isfinite(got) && isfinite(d64)) ++l_nf;
                if (diff > l_diff || isnan(diff)) l_diff = isnan(diff) ? INFINITY : diff;
                if (fabs(d64) > l_d) l_d = fabs(d64);
                if (fabs(crv - d64) > l_gap) l_gap = fabs(crv - d64);
                if (!(got == crv)) ++l_bad;
                ++l_cmp;
            }
        }
#pragma omp critical
        {
            if (l_diff > max_diff) max_diff = l_diff;
            if (l_d > max_d) max_d = l_d;
            if (l_gap > max_gap) max_gap = l_gap;
            n_cmp += l_cmp;
            n_bad += l_bad;
            n_nonfinite += l_nf;
        }
    }
    stats[0] = max_diff;
    stats[1] = max_d;
    stats[2] = max_gap;
    counts[0] = n_cmp;
    counts[1] = n_bad;
    counts[2] = n_nonfinite;
}

/* Range partials of the scaled row (m = max s x, s = sum exp(s x - m)). */
void oracle_range_partials(const void* x, int dtype, int64_t n, int64_t v, int64_t ld,
                              int64_t w, int64_t k, double s, double* pm, double* ps) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        for (int64_t j = 0; j < k; ++j) {
            int64_t c0 = j * w, c1 = (j + 1) * w;
            if (c0 > v) c0 = v;
            if (c1 > v) c1 = v;
            range_max_sumexp(x, dtype, ld, t, c0, c1, s, &pm[t * k + j], &ps[t * k + j]);
        }
    }
}

/* ---- fused LM head + logp ------------------------------------------------- */

/* linear_logp (named in RL-Kernel PR #495, Summary, among the ops that PR
 * leaves alone; the pages give no formula): the logits are the LM-head
 * contraction z[t, j] = sum_k h[t, k] w[j, k] of the BF16 hidden states
 * h [n, d] (row stride ldh) with the BF16 weight rows w [v, d] (row stride
 * ldw), and the selected-token logprob of issue #241 (Background, Goal) is
 * taken of s z.  Per row, in double: every z_j (a product of two BF16 values
 * is exact in double), then the plain two-pass LSE = M + log sum exp(s z_j - M),
 * logp = s z_y - LSE for active rows, else 0.  bound[t] (if not NULL) is
 * max_j sum_k |h[t, k] w[j, k]|: the scale of the rounding error of any
 * binary32 evaluation of the row's logits, for the tests' tolerance. */
void oracle_linear_logp(const uint16_t* h, int64_t ldh, const uint16_t* w, int64_t ldw,
                        int64_t n, int64_t d, int64_t v, const int64_t* y, int64_t ignore_index,
                        const uint8_t* mask, double s, double* logp, double* lse, double* bound) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n; ++t) {
        double* hz = (double*)malloc(sizeof(double) * (size_t)(d + v));
        double* z = hz + d;
        for (int64_t k = 0; k < d; ++k) hz[k] = bf16_bits_to_double(h[t * ldh + k]);
        double babs = 0.0;
        for (int64_t j = 0; j < v; ++j) {
            const uint16_t* wj = w + j * ldw;
            double acc = 0.0, aabs = 0.0;
            for (int64_t k = 0; k < d; ++k) {
                const double p = hz[k] * bf16_bits_to_double(wj[k]);
                acc += p;
                aabs += fabs(p);
            }
            z[j] = acc;
            if (aabs > babs) babs = aabs;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < v; ++j)
            if (s * z[j] > m) m = s * z[j];
        double acc = 0.0;
        for (int64_t j = 0; j < v; ++j) acc += exp(s * z[j] - m);
        const double l = m + log(acc);
        lse[t] = l;
        logp[t] = row_active(y, mask, t, v, ignore_index) ? s * z[y[t]] - l : 0.0;
        if (bound) bound[t] = babs;
        free(hz);
    }
}

/* Backward of the fused LM head: the gradient of sum_t g_t logp_t through
 * z = H W^T, i.e. the backward of RL-Kernel PR #495 (Summary item 2),
 * dZ[t, j] = s g_t (onehot(y_t)[j] - exp(s z_tj - LSE_t)) for active rows
 * (0 otherwise; the target column as -s g_t expm1(s z_ty - LSE_t)), followed
 * by the chain rule through the contraction: dH = dZ W, dW = dZ^T H.  With
 * round_dz, every dZ value is first rounded to BF16, as the method writes
 * dlogits in BF16.  dz [n, v] (optional), dh [n, d], dw [v, d] are dense
 * row-major doubles; everything is computed in double. */
void oracle_linear_backward(const uint16_t* h, int64_t ldh, const uint16_t* w, int64_t ldw,
                            int64_t n, int64_t d, int64_t v, const int64_t* y, int64_t ignore_index,
                            const uint8_t* mask, double s, const float* g, int round_dz,
                            double* dz_out, double* dh, double* dw) {
    double* dz = dz_out ? dz_out : (double*)malloc(sizeof(double) * (size_t)(n * v));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n; ++t) {
        double* row = dz + t * v;
        if (!row_active(y, mask, t, v, ignore_index)) {
            for (int64_t j = 0; j < v; ++j) row[j] = 0.0;
            continue;
        }
        double* hz = (double*)malloc(sizeof(double) * (size_t)d);
        for (int64_t k = 0; k < d; ++k) hz[k] = bf16_bits_to_double(h[t * ldh + k]);
        for (int64_t j = 0; j < v; ++j) {
            const uint16_t* wj = w + j * ldw;
            double acc = 0.0;
            for (int64_t k = 0; k < d; ++k) acc += hz[k] * bf16_bits_to_double(wj[k]);
            row[j] = s * acc;                         /* s z */
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < v; ++j)
            if (row[j] > m) m = row[j];
        double sum = 0.0;
        for (int64_t j = 0; j < v; ++j) sum += exp(row[j] - m);
        const double l = m + log(sum);
        const double sg = s * (double)g[t];
        for (int64_t j = 0; j < v; ++j)
            row[j] = (j == y[t]) ? -sg * expm1(row[j] - l) : -sg * exp(row[j] - l);
        if (round_dz)
            for (int64_t j = 0; j < v; ++j) row[j] = bf16_bits_to_double(oracle_round_bf16(row[j]));
        free(hz);
    }
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        for (int64_t k = 0; k < d; ++k) dh[t * d + k] = 0.0;
        for (int64_t j = 0; j < v; ++j) {
            const double z = dz[t * v + j];
            if (z == 0.0) continue;
            const uint16_t* wj = w + j * ldw;
            for (int64_t k = 0; k < d; ++k) dh[t * d + k] += z * bf16_bits_to_double(wj[k]);
        }
    }
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < v; ++j) {
        for (int64_t k = 0; k < d; ++k) dw[j * d + k] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            const double z = dz[t * v + j];
            if (z == 0.0) continue;
            for (int64_t k = 0; k < d; ++k) dw[j * d + k] += z * bf16_bits_to_double(h[t * ldh + k]);
        }
    }
    if (!dz_out) free(dz);
}

/* ---- GRPO loss on the logp path -------------------------------------------- */

/* Issue #241 PR 5 names the objective (ratio, clip, KL, advantage) and three
 * normalisers without formulas; this is the standard clipped-surrogate form:
 * per active token t (mask byte nonzero, or every token when mask is NULL)
 *   r_t  = exp(logp_t - old_t)
 *   pg_t = max(-A_t r_t, -A_t clip(r_t, 1 - eps_lo, 1 + eps_hi))
 *   kl_t = exp(ref_t - logp_t) - (ref_t - logp_t) - 1   (only if ref != NULL)
 *   l_t  = pg_t + beta kl_t
 * and the loss over sequences s = [cu[s], cu[s+1]) (n_s active tokens,
 * S' = sequences with n_s > 0):
 *   mode 0 token mean:               L = sum_t l_t / D,  D = sum_s n_s
 *   mode 1 sequence mean of token means: L = (1/S') sum_s (sum_{t in s} l_t) / n_s
 *   mode 2 sequence mean of token sums:  L = (1/S') sum_s sum_{t in s} l_t
 * A positive `normalizer` replaces D (mode 0) or S' (modes 1, 2), as when the
 * count is global across micro-batches.  With cu == NULL the whole batch is
 * one sequence.  The gradient with respect to logp_t is
 *   g_t = w_t (dpg_t + beta (1 - exp(ref_t - logp_t))),
 *   dpg_t = -A_t r_t when the unclipped term is the max (ties included), else 0,
 *   w_t = 1/D, 1/(S' n_s) or 1/S'; 0 for inactive tokens.
 * Everything in double. */
void oracle_grpo_loss(const double* logp, const double* old, const double* ref,
                      const double* adv, const uint8_t* mask, const int64_t* cu, int64_t nseq,
                      int64_t n, int mode, double eps_lo, double eps_hi, double beta,
                      double normalizer, double* loss, double* g) {
    int64_t one_cu[2] = {0, n};
    if (cu == 0) {
        cu = one_cu;
        nseq = 1;
    }
    double tot = 0.0, d_tok = 0.0, s_act = 0.0, seq_terms = 0.0;
    /* a token in no sequence takes part in no term: gradient 0 */
    for (int64_t t = 0; t < n; ++t) g[t] = 0.0;
    for (int64_t s = 0; s < nseq; ++s) {
        double sum = 0.0, cnt = 0.0;
        for (int64_t t = cu[s]; t < cu[s + 1]; ++t) {
            if (mask && !mask[t]) continue;
            double r = exp(logp[t] - old[t]);
            double rc = r < 1.0 - eps_lo ? 1.0 - eps_lo : (r > 1.0 + eps_hi ? 1.0 + eps_hi : r);
            double p1 = -adv[t] * r, p2 = -adv[t] * rc;
            double l = p1 >= p2 ? p1 : p2;
            if (ref) {
                double dlt = ref[t] - logp[t];
                l += beta * (exp(dlt) - dlt - 1.0);
            }
            sum += l;
            cnt += 1.0;
        }
        tot += sum;
        d_tok += cnt;
        if (cnt > 0) {
            s_act += 1.0;
            seq_terms += (mode == 1) ? sum / cnt : sum;
        }
    }
    double den = (mode == 0) ? d_tok : s_act;
    if (normalizer > 0) den = normalizer;
    double num = (mode == 0) ? tot : seq_terms;
    *loss = den > 0 ? num / den : 0.0;
    for (int64_t s = 0; s < nseq; ++s) {
        double cnt = 0.0;
        for (int64_t t = cu[s]; t < cu[s + 1]; ++t) cnt += (mask && !mask[t]) ? 0.0 : 1.0;
        for (int64_t t = cu[s]; t < cu[s + 1]; ++t) {
            if ((mask && !mask[t]) || den <= 0) {
                g[t] = 0.0;
                continue;
            }
            double w = (mode == 1) ? 1.0 / (den * cnt) : 1.0 / den;
            double r = exp(logp[t] - old[t]);
            double rc = r < 1.0 - eps_lo ? 1.0 - eps_lo : (r > 1.0 + eps_hi ? 1.0 + eps_hi : r);
            double p1 = -adv[t] * r, p2 = -adv[t] * rc;
            double d = p1 >= p2 ? -adv[t] * r : 0.0;
            if (ref) d += beta * (1.0 - exp(ref[t] - logp[t]));
            g[t] = w * d;
        }
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

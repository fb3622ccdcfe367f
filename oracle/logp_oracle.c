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
 * Everything is computed in IEEE double from the exact BF16 inputs with a
 * plain two-pass log-sum-exp.  Compile with -ffp-contract=off so that x86
 * and Arm hosts round identically.
 */
#include <math.h>
#include <stdint.h>
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

/* ---- row log-sum-exp ----------------------------------------------------- */

/* A row is active when its target names a real vocabulary column and is not
 * the ignore index (PR #495, Behavior changes: out-of-range targets). */
static int row_active(int64_t y, int64_t v, int64_t ignore_index) {
    return y >= 0 && y < v && y != ignore_index;
}

/* Plain two-pass log-sum-exp over columns [c0, c1) of one row:
 * m = max x, lse = m + log(sum exp(x - m)).  An all -inf range gives
 * m = -inf and lse = -inf (the identity partial's log-sum-exp). */
static void range_max_sumexp(const uint16_t* xr, int64_t c0, int64_t c1,
                             double* m_out, double* s_out) {
    double m = -INFINITY;
    for (int64_t c = c0; c < c1; ++c) {
        double x = bf16_bits_to_double(xr[c]);
        if (x > m) m = x;
    }
    double s = 0.0;
    if (m != -INFINITY) {
        for (int64_t c = c0; c < c1; ++c) {
            double x = bf16_bits_to_double(xr[c]);
            if (x != -INFINITY) s += exp(x - m);
        }
    }
    *m_out = m;
    *s_out = s;
}

static double row_lse(const uint16_t* xr, int64_t v) {
    double m, s;
    range_max_sumexp(xr, 0, v, &m, &s);
    if (m == -INFINITY) return -INFINITY;
    return m + log(s);
}

/* ---- forward: logp and lse ----------------------------------------------- */

/* logp[t] = x[t, y_t] - LSE_t for active rows, 0 otherwise; lse[t] = LSE_t
 * for every row (issue #241 Background; PR #495 Behavior changes). */
void oracle_forward(const uint16_t* x, int64_t n, int64_t v, int64_t ld,
                    const int64_t* y, int64_t ignore_index,
                    double* logp, double* lse) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* xr = x + t * ld;
        double l = row_lse(xr, v);
        lse[t] = l;
        logp[t] = row_active(y[t], v, ignore_index)
                      ? bf16_bits_to_double(xr[y[t]]) - l
                      : 0.0;
    }
}

/* ---- backward ------------------------------------------------------------ */

/* One gradient element of an active row: d = g * (onehot - softmax), with the
 * softmax taken as exp(x - LSE) (PR #495 Summary item 2).  On the target
 * column 1 - exp(u) is written as -expm1(u), the same quantity without the
 * cancellation when the target's probability is near 1. */
static double grad_elem(double x, double l, double g, int on_target) {
    double u = x - l;
    return on_target ? -g * expm1(u) : -g * exp(u);
}

/* Dense FP64 gradient for small shapes: d[t*ld_d + c].  Inactive rows are
 * exactly zero. */
void oracle_backward(const uint16_t* x, int64_t n, int64_t v, int64_t ld,
                     const int64_t* y, int64_t ignore_index, const float* g,
                     double* d, int64_t ld_d) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* xr = x + t * ld;
        double* dr = d + t * ld_d;
        if (!row_active(y[t], v, ignore_index)) {
            for (int64_t c = 0; c < v; ++c) dr[c] = 0.0;
            continue;
        }
        double l = row_lse(xr, v);
        double gt = (double)g[t];
        for (int64_t c = 0; c < v; ++c)
            dr[c] = grad_elem(bf16_bits_to_double(xr[c]), l, gt, c == y[t]);
    }
}

/* Streaming comparison of a BF16 gradient against the FP64 gradient, one row
 * at a time, never holding an FP64 [n, v] array.  stats (doubles):
 *   [0] max |dl - d64|            [1] max |d64|
 *   [2] max |round_bf16(d64) - d64|   (the error a correctly rounded result has)
 * counts (int64):
 *   [0] elements compared   [1] elements whose bits differ from round_bf16(d64)
 *   [2] elements that are NaN/inf in dl where d64 is finite
 * Values are compared as numbers, so +0 and -0 count as equal. */
void oracle_backward_compare(const uint16_t* x, int64_t n, int64_t v, int64_t ld,
                             const int64_t* y, int64_t ignore_index,
                             const float* g, const uint16_t* dl, int64_t ld_out,
                             double* stats, int64_t* counts) {
    double max_diff = 0.0, max_d = 0.0, max_gap = 0.0;
    int64_t n_cmp = 0, n_bad = 0, n_nonfinite = 0;
#pragma omp parallel
    {
        double l_diff = 0.0, l_d = 0.0, l_gap = 0.0;
        int64_t l_cmp = 0, l_bad = 0, l_nf = 0;
#pragma omp for schedule(static)
        for (int64_t t = 0; t < n; ++t) {
            const uint16_t* xr = x + t * ld;
            const uint16_t* gr = dl + t * ld_out;
            int act = row_active(y[t], v, ignore_index);
            double l = act ? row_lse(xr, v) : 0.0;
            double gt = (double)g[t];
            for (int64_t c = 0; c < v; ++c) {
                double d64 = act ? grad_elem(bf16_bits_to_double(xr[c]), l, gt, c == y[t]) : 0.0;
                uint16_t cr = oracle_round_bf16(d64);
                double crv = bf16_bits_to_double(cr);
                double got = bf16_bits_to_double(gr[c]);
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

/* ---- vocab partials and their merge ---------------------------------------- */

/* Per-range partials (issue #241, PR 3 bullets): for each row and each of k
 * consecutive column ranges of width w (the last ones clipped at v, empty
 * ones giving the identity (-inf, 0)), m = max x and s = sum exp(x - m). */
void oracle_range_partials(const uint16_t* x, int64_t n, int64_t v, int64_t ld,
                           int64_t w, int64_t k, double* pm, double* ps) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t* xr = x + t * ld;
        for (int64_t j = 0; j < k; ++j) {
            int64_t c0 = j * w, c1 = (j + 1) * w;
            if (c0 > v) c0 = v;
            if (c1 > v) c1 = v;
            range_max_sumexp(xr, c0, c1, &pm[t * k + j], &ps[t * k + j]);
        }
    }
}

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

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

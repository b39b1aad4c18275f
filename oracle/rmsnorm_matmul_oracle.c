/*
 * CPU oracle for the fused RMSNorm + matmul (test infrastructure only).
 *
 * Page: matmul_rms_norm.wgsl (meganeura 0.2.0), header comment and the
 * prologue / A-tile load of its compute entry point.  It defines
 *
 *     C = RmsNorm(X, W_norm) x W_proj,   X [M, K], W_proj [K, N], W_norm [K],
 *     RmsNorm(X, W_norm)[i, t] = X[i, t] * r[i] * W_norm[t],
 *     r[i] = 1 / sqrt( (sum over t of X[i, t]^2) / K + eps ),
 *
 * all matrices row-major, C [M, N].  These functions restate that definition
 * with plain double-precision loops in the order the page states it (row
 * scale first, then the product); nothing is blocked, fused or reordered.
 * Nothing here is shared with the CUDA library, and the library never calls
 * it.  Pins: tests/test_rmsnorm_oracle_pins.py (hand-worked golden values,
 * closed forms, scale and sign invariants, torch's own rms_norm, planted
 * mutants of this file).
 */
#include <math.h>
#include <stdint.h>

/* r[i] for every row: the page's prologue (sum of squares over K, divided by
 * K, plus eps, reciprocal square root).  Returns 0, or -1 for a bad shape. */
int oracle_rms_rows_f64(const double *x, double *r, int m, int k, double eps) {
    if (m < 0 || k <= 0) return -1;
    for (int i = 0; i < m; ++i) {
        double ss = 0.0;
        for (int t = 0; t < k; ++t) ss += x[(int64_t)i * k + t] * x[(int64_t)i * k + t];
        r[i] = 1.0 / sqrt(ss / (double)k + eps);
    }
    return 0;
}

/* The normalised operand A[i, t] = X[i, t] * r[i] * W_norm[t] (the page's
 * A-tile load, over the whole matrix). */
int oracle_rms_normalize_f64(const double *x, const double *w_norm, double *a, int m, int k, double eps) {
    if (m < 0 || k <= 0) return -1;
    for (int i = 0; i < m; ++i) {
        double ss = 0.0;
        for (int t = 0; t < k; ++t) ss += x[(int64_t)i * k + t] * x[(int64_t)i * k + t];
        const double r = 1.0 / sqrt(ss / (double)k + eps);
        for (int t = 0; t < k; ++t) a[(int64_t)i * k + t] = x[(int64_t)i * k + t] * r * w_norm[t];
    }
    return 0;
}

/* C [M, N] = A x W_proj with A the normalised operand above. */
int oracle_rmsnorm_matmul_f64(const double *x, const double *w_norm, const double *w_proj, double *c,
                              int m, int n, int k, double eps) {
    if (m < 0 || n < 0 || k <= 0) return -1;
    for (int i = 0; i < m; ++i) {
        double ss = 0.0;
        for (int t = 0; t < k; ++t) ss += x[(int64_t)i * k + t] * x[(int64_t)i * k + t];
        const double r = 1.0 / sqrt(ss / (double)k + eps);
        for (int j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int t = 0; t < k; ++t)
                acc += (x[(int64_t)i * k + t] * r * w_norm[t]) * w_proj[(int64_t)t * n + j];
            c[(int64_t)i * n + j] = acc;
        }
    }
    return 0;
}

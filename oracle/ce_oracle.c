/*
 * Softmax cross-entropy oracle: plain fp64 loops on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header or constant with the CUDA path.
 *
 * What it computes (the fused loss + gradient of rumus milestone M7a, "GPU-fused
 * Cross-Entropy Loss with Log-Sum-Exp stability ... gradient pre-computed during
 * forward", rumus project page; the per-row steps of Pass 1 of the
 * cross_entropy.wgsl source page of rumus 0.1.1), for every row b of a
 * row-major logits matrix z[B][C] with integer target t_b:
 *
 *   Step 1 (max logit)            m_b   = max_c z[b][c]
 *   Step 2 (sum of exp(z - max))  S_b   = sum_c exp(z[b][c] - m_b)
 *   Step 3 (per-batch loss)       l_b   = log(S_b) - (z[b][t_b] - m_b)
 *   Step 4 (gradient)             g[b][c] = (exp(z[b][c] - m_b) / S_b - [c == t_b]) / B
 *   Pass 2 (reduce to a scalar)   L     = (sum_b l_b) / B
 *
 * Readings where the pages leave a step open:
 *   - the max starts at -infinity (the shader starts at -3.402823e+38; equal
 *     for every finite input);
 *   - targets are int32 class indices (the shader stores them as f32);
 *   - a target outside [0, C) is an error: that row's loss is NaN (so L is
 *     NaN) and its gradient is softmax/B with no one-hot term;
 *   - 1/B is applied once to the sum of the row losses (the shader divides each
 *     row's loss by B before summing; identical in exact arithmetic);
 *   - bf16 and f16 logits are widened exactly to fp64 before any arithmetic
 *     (f16 from the binary16 definition: rumus milestone M11 names f16
 *     storage with f32 accumulation and fixes nothing more);
 *   - the reductions sum and none, and an upstream gradient u (rumus M7a:
 *     the backward scales the precomputed gradient by the upstream value):
 *     the sum reduction's gradient has no 1/B, none's is d l_b / d z_b, and
 *     u multiplies the gradient (a scalar, or one value per row for none);
 *   - the row softmax of rumus milestone M8c (forward and backward kernels,
 *     log-sum-exp stable; no formulas printed): p = exp(z - m) / sum exp(z - m)
 *     and dx = p * (dy - sum_c p_c dy_c), with p and dy read in the logits'
 *     element type.
 *
 * Accumulation is in double, in class order within a row and row order for L.
 * Rows are independent and may run on several OpenMP threads; each row's
 * result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F16 2

/* IEEE binary16 bits to double, from the format's definition: sign bit,
 * 5 exponent bits with bias 15, 10 fraction bits; exponent 0 is subnormal
 * (2^-14 * f/1024), exponent 31 is infinity (f = 0) or NaN. */
static double oracle_half(uint16_t h) {
    const int sign = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* Widen one element of the logits to double (bf16 -> fp32 and f16 -> double
 * are exact). */
static double oracle_z(const void *logits, int dtype, int64_t i) {
    if (dtype == ORACLE_F32) return (double)((const float *)logits)[i];
    if (dtype == ORACLE_F16) return oracle_half(((const uint16_t *)logits)[i]);
    uint32_t bits = ((uint32_t)((const uint16_t *)logits)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* One row: the four steps of Pass 1.  grad_row may be NULL (loss only);
 * factor multiplies the gradient (1/B for the batch mean). */
static double oracle_row(const void *logits, int dtype, int64_t b, int64_t C,
                         int32_t t, double factor, double *grad_row) {
    const int64_t row_start = b * C;
    int target_ok = (t >= 0 && (int64_t)t < C);

    double m = -INFINITY; /* Step 1 */
    for (int64_t c = 0; c < C; ++c) {
        double z = oracle_z(logits, dtype, row_start + c);
        if (z > m) m = z;
    }

    double s = 0.0; /* Step 2 */
    for (int64_t c = 0; c < C; ++c) s += exp(oracle_z(logits, dtype, row_start + c) - m);

    double loss = NAN; /* Step 3 */
    if (target_ok) loss = log(s) - (oracle_z(logits, dtype, row_start + t) - m);

    if (grad_row) { /* Step 4 */
        for (int64_t c = 0; c < C; ++c) {
            double p = exp(oracle_z(logits, dtype, row_start + c) - m) / s;
            double one_hot = (target_ok && c == (int64_t)t) ? 1.0 : 0.0;
            grad_row[c] = (p - one_hot) * factor;
        }
    }
    return loss;
}

/* Number of threads the oracle's parallel loops use. */
int ce_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ce_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Per-row losses and (optionally) gradients for a list of rows.
 *   logits   [B][C] row-major, fp32 (dtype 0), bf16 bit patterns (dtype 1) or
 *            IEEE binary16 bit patterns (dtype 2)
 *   targets  [B] int32
 *   rows     row indices to evaluate (NULL: all rows 0..B-1, nrows must be B)
 *   loss     [nrows] out, l_b of each listed row
 *   grad     [nrows][C] out in fp64, or NULL
 * Returns 0, or -1 on a bad argument.
 */
int ce_oracle_rows(const void *logits, int dtype, const int32_t *targets, int64_t B,
                   int64_t C, const int64_t *rows, int64_t nrows, double *loss,
                   double *grad) {
    if (!logits || !targets || !loss || B <= 0 || C <= 0 || nrows < 0) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
    if (!rows && nrows != B) return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= B)) return -1;
    const double inv_b = 1.0 / (double)B;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t b = rows ? rows[i] : i;
        loss[i] = oracle_row(logits, dtype, b, C, targets[b], inv_b,
                             grad ? grad + i * C : (double *)0);
    }
    return 0;
}

/* Pass 2: L = (sum_b l_b) / B, summed in row order. */
double ce_oracle_batch_loss(const double *loss_rows, int64_t B) {
    double s = 0.0;
    for (int64_t b = 0; b < B; ++b) s += loss_rows[b];
    return s / (double)B;
}

/*
 * The reductions and the upstream gradient.  The rumus project page's backward
 * for this loss (milestone M7a) multiplies the gradient precomputed in the
 * forward pass by the upstream gradient; written out for each reduction of
 * the row losses l_b:
 *   mean (0):  L = (1/B) sum_b l_b   dL/dz[b][c]     = (p[b][c] - [c == t_b]) / B
 *   sum  (1):  L = sum_b l_b         dL/dz[b][c]     = p[b][c] - [c == t_b]
 *   none (2):  L_b = l_b             dL_b/dz[b][c]   = p[b][c] - [c == t_b]
 * and with an upstream gradient u (one value for mean and sum, u_b per row
 * for none; NULL means 1) the gradient returned is u * dL/dz.
 *   upstream  NULL, [1] (mean, sum) or [B] (none), in fp64
 * Otherwise as ce_oracle_rows.  Returns 0, or -1 on a bad argument.
 */
int ce_oracle_rows_ex(const void *logits, int dtype, const int32_t *targets, int64_t B,
                      int64_t C, int reduction, const double *upstream, const int64_t *rows,
                      int64_t nrows, double *loss, double *grad) {
    if (!logits || !targets || !loss || B <= 0 || C <= 0 || nrows < 0) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
    if (reduction < 0 || reduction > 2) return -1;
    if (!rows && nrows != B) return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= B)) return -1;
    const double base = reduction == 0 ? 1.0 / (double)B : 1.0;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t b = rows ? rows[i] : i;
        double u = 1.0;
        if (upstream) u = reduction == 2 ? upstream[b] : upstream[0];
        loss[i] = oracle_row(logits, dtype, b, C, targets[b], base * u,
                             grad ? grad + i * C : (double *)0);
    }
    return 0;
}

/* Pass 2 for a reduction: (sum_b l_b) / B for the mean, sum_b l_b for the sum,
 * summed in row order. */
double ce_oracle_reduce(const double *loss_rows, int64_t B, int reduction) {
    double s = 0.0;
    for (int64_t b = 0; b < B; ++b) s += loss_rows[b];
    return reduction == 0 ? s / (double)B : s;
}

/*
 * Row-wise softmax, forward and backward (rumus project page, milestone M8c:
 * row-wise softmax with log-sum-exp stability, forward and backward kernels).
 *   forward   p[b][c] = exp(z[b][c] - m_b) / sum_c' exp(z[b][c'] - m_b)
 *   backward  dx[b][c] = p[b][c] * (dy[b][c] - sum_c' p[b][c'] dy[b][c'])
 * in fp64, inputs widened exactly from `dtype`; `rows` as in ce_oracle_rows;
 * out is [nrows][C].  Returns 0, or -1 on a bad argument.
 */
int ce_oracle_softmax(const void *logits, int dtype, int64_t B, int64_t C, const int64_t *rows,
                      int64_t nrows, double *out) {
    if (!logits || !out || B <= 0 || C <= 0 || nrows < 0) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
    if (!rows && nrows != B) return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= B)) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t row_start = (rows ? rows[i] : i) * C;
        double m = -INFINITY;
        for (int64_t c = 0; c < C; ++c) {
            double z = oracle_z(logits, dtype, row_start + c);
            if (z > m) m = z;
        }
        double s = 0.0;
        for (int64_t c = 0; c < C; ++c) s += exp(oracle_z(logits, dtype, row_start + c) - m);
        for (int64_t c = 0; c < C; ++c)
            out[i * C + c] = exp(oracle_z(logits, dtype, row_start + c) - m) / s;
    }
    return 0;
}

int ce_oracle_softmax_bwd(const void *probs, const void *dy, int dtype, int64_t B, int64_t C,
                          const int64_t *rows, int64_t nrows, double *out) {
    if (!probs || !dy || !out || B <= 0 || C <= 0 || nrows < 0) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
    if (!rows && nrows != B) return -1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= B)) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t row_start = (rows ? rows[i] : i) * C;
        double dot = 0.0;
        for (int64_t c = 0; c < C; ++c)
            dot += oracle_z(probs, dtype, row_start + c) * oracle_z(dy, dtype, row_start + c);
        for (int64_t c = 0; c < C; ++c)
            out[i * C + c] = oracle_z(probs, dtype, row_start + c) *
                             (oracle_z(dy, dtype, row_start + c) - dot);
    }
    return 0;
}

/* Narrow a double to fp32 and then to bf16 (round to nearest even each time). */
static uint16_t oracle_to_bf16(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/*
 * The whole forward + gradient, as a user of the path would call it: the batch
 * loss L and the gradient written in the logits' own element type (fp32, or
 * bf16 narrowed through fp32).  Used to time the oracle; parity checks use the
 * fp64 values of ce_oracle_rows.  row_scratch holds B doubles.
 */
int ce_oracle_fwd_bwd(const void *logits, int dtype, const int32_t *targets, int64_t B,
                      int64_t C, double *loss_out, void *grad_out, double *row_scratch) {
    if (!logits || !targets || !loss_out || !grad_out || !row_scratch || B <= 0 || C <= 0)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
    const double inv_b = 1.0 / (double)B;
    int bad = 0;
#pragma omp parallel
    {
        double *g = 0;
        /* one fp64 row buffer per thread, on the stack for modest C */
        double small[4096];
        double *heap = 0;
        if (C <= 4096) {
            g = small;
        } else {
            heap = (double *)malloc((size_t)C * sizeof(double));
            g = heap;
        }
        if (!g) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t b = 0; b < B; ++b) {
            if (!g) continue;
            row_scratch[b] = oracle_row(logits, dtype, b, C, targets[b], inv_b, g);
            if (dtype == ORACLE_F32) {
                float *o = (float *)grad_out + b * C;
                for (int64_t c = 0; c < C; ++c) o[c] = (float)g[c];
            } else {
                uint16_t *o = (uint16_t *)grad_out + b * C;
                for (int64_t c = 0; c < C; ++c) o[c] = oracle_to_bf16(g[c]);
            }
        }
        free(heap);
    }
    if (bad) return -1;
    *loss_out = ce_oracle_batch_loss(row_scratch, B);
    return 0;
}

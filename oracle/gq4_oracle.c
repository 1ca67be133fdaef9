/*
 * gq4_oracle.c -- plain CPU oracle for the int4 group-quantized matvec family.
 *
 * TEST INFRASTRUCTURE ONLY (see gq4_oracle.h).  Written for a reader who
 * checks it against the definitions by eye: no blocking, no fusion, no
 * reordering.  Sums run over k in increasing order in double precision.
 * Build with -ffp-contract=off so that no step is fused into an FMA.
 *
 * Parity pins (checked by tests/test_oracle_pins.py, not by this file):
 *   unpack      -- an independent byte-view unpack, fixed words, pack round trip
 *   dequant     -- one-hot activations return w(n,k) exactly
 *   dot         -- exact rational brute force on dyadic inputs
 *   zero        -- all codes equal to integer zeros give exactly 0
 *   quad        -- concatenated outputs equal the unsplit matvec
 *   norm        -- closed form on constant input, scale invariance, f32 residual
 *   gated       -- all-ones up matrix gives sum(a), zero gate gives 0, composition
 *   gated input -- sigmoid(0) halves, saturated gates pass or scale the input
 *                  exactly, silu(0) gives exactly 0
 *   quantize    -- values on a 16-level grid come back exactly; every code is
 *                  the nearest level (brute force over the 16); error within
 *                  half a step; both ends of every group are used
 *   MLX         -- a worked word with scale 1/2 and bias -4; conversion agrees
 *                  with the page's dequant within rounding; degenerate groups
 *                  reproduce the bias exactly
 *   embedding   -- rows equal a numpy binary32 dequant of byte-view codes of
 *                  the chosen rows; out-of-range ids give NaN rows
 */
#include "gq4_oracle.h"

#include <float.h>
#include <math.h>
#include <stddef.h>
#include <stdlib.h>

/* The quantizer decides integer codes in binary32: float expressions must be
 * evaluated in float, one rounding per operation. */
#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs FLT_EVAL_METHOD == 0"
#endif

static int shape_ok(int M, int K, int N, int gs)
{
    if (M <= 0 || K <= 0 || N <= 0 || gs <= 0) return 0;
    if (K % 8 != 0) return 0;      /* a column is K/8 whole words */
    if (K % gs != 0) return 0;     /* a column is K/gs whole groups */
    return 1;
}

/* Element k of column n: word k/8 of the column, nibble k%8, low nibble
 * first (WGSL_QUAD_MATVEC_INT4 main loop: `packed & 0xF`, then `>> 4`, ...). */
int gq4o_nibble(const uint32_t *Bq, int K, int n, int k)
{
    const uint32_t word = Bq[(size_t)n * (size_t)(K / 8) + (size_t)(k / 8)];
    return (int)((word >> (4 * (k % 8))) & 0xFu);
}

int gq4o_unpack(int K, int N, const uint32_t *Bq, uint8_t *q)
{
    if (!shape_ok(1, K, N, 8) || !Bq || !q) return -1;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            q[(size_t)n * K + k] = (uint8_t)gq4o_nibble(Bq, K, n, k);
    return 0;
}

int gq4o_pack(int K, int N, const uint8_t *q, uint32_t *Bq)
{
    if (!shape_ok(1, K, N, 8) || !Bq || !q) return -1;
    const size_t words = (size_t)N * (size_t)(K / 8);
    for (size_t i = 0; i < words; ++i) Bq[i] = 0u;
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            const uint32_t code = (uint32_t)q[(size_t)n * K + k];
            if (code > 15u) return -1;
            Bq[(size_t)n * (K / 8) + k / 8] |= code << (4 * (k % 8));
        }
    }
    return 0;
}

/* Group of element k along its column (WGSL main loop: one scale and one
 * zero per group_size consecutive k of a column, row n*G + k/gs). */
static size_t group_index(int K, int gs, int n, int k)
{
    return (size_t)n * (size_t)(K / gs) + (size_t)(k / gs);
}

/* w(n,k) = (q - zero) * scale.  In double, q - zero is exact (q is a small
 * integer, zero a binary32 value) and so is the product with a binary32
 * scale (24 + 24 significant bits fit in 53). */
static double weight(int K, int gs, const uint32_t *Bq, const float *scales,
                     const float *zeros, int n, int k)
{
    const size_t g = group_index(K, gs, n, k);
    const double q = (double)gq4o_nibble(Bq, K, n, k);
    return (q - (double)zeros[g]) * (double)scales[g];
}

int gq4o_dequant_f64(int K, int N, int gs, const uint32_t *Bq,
                     const float *scales, const float *zeros, double *W)
{
    if (!shape_ok(1, K, N, gs) || !Bq || !scales || !zeros || !W) return -1;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            W[(size_t)n * K + k] = weight(K, gs, Bq, scales, zeros, n, k);
    return 0;
}

int gq4o_dequant_f32(int K, int N, int gs, const uint32_t *Bq,
                     const float *scales, const float *zeros, float *W)
{
    if (!shape_ok(1, K, N, gs) || !Bq || !scales || !zeros || !W) return -1;
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            const size_t g = group_index(K, gs, n, k);
            volatile float t = (float)gq4o_nibble(Bq, K, n, k) - zeros[g];
            volatile float w = t * scales[g];
            W[(size_t)n * K + k] = w;
        }
    }
    return 0;
}

double gq4o_dot(int K, int gs, const double *a, const uint32_t *Bq,
                const float *scales, const float *zeros, int n, double *S)
{
    double sum = 0.0, abs_sum = 0.0;
    for (int k = 0; k < K; ++k) {
        const double term = a[k] * weight(K, gs, Bq, scales, zeros, n, k);
        sum += term;
        abs_sum += fabs(term);
    }
    if (S) *S = abs_sum;
    return sum;
}

int gq4o_matvec_cols(int M, int K, int gs, const double *a,
                     const uint32_t *Bq, const float *scales,
                     const float *zeros, int ncols, const int *cols,
                     double *C, double *S)
{
    if (!shape_ok(M, K, 1, gs) || ncols < 0 || !a || !Bq || !scales ||
        !zeros || (ncols > 0 && (!cols || !C)))
        return -1;
    for (int m = 0; m < M; ++m) {
        for (int j = 0; j < ncols; ++j) {
            if (cols[j] < 0) return -1;
            double s_abs = 0.0;
            C[(size_t)m * ncols + j] = gq4o_dot(K, gs, a + (size_t)m * K, Bq,
                                                scales, zeros, cols[j], &s_abs);
            if (S) S[(size_t)m * ncols + j] = s_abs;
        }
    }
    return 0;
}

/* Dot product of one f32 activation row with column n. */
static double dot_f32(int K, int gs, const float *a, const uint32_t *Bq,
                      const float *scales, const float *zeros, int n,
                      double *S)
{
    double sum = 0.0, abs_sum = 0.0;
    for (int k = 0; k < K; ++k) {
        const double term =
            (double)a[k] * weight(K, gs, Bq, scales, zeros, n, k);
        sum += term;
        abs_sum += fabs(term);
    }
    if (S) *S = abs_sum;
    return sum;
}

int gq4o_matvec(int M, int K, int N, int gs, const float *A,
                const uint32_t *Bq, const float *scales, const float *zeros,
                double *C, double *S)
{
    if (!shape_ok(M, K, N, gs) || !A || !Bq || !scales || !zeros || !C)
        return -1;
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            double s_abs = 0.0;
            C[(size_t)m * N + n] = dot_f32(K, gs, A + (size_t)m * K, Bq,
                                           scales, zeros, n, &s_abs);
            if (S) S[(size_t)m * N + n] = s_abs;
        }
    }
    return 0;
}

/* Quad routing (WGSL_QUAD_MATVEC_INT4 epilogue): the matvec runs over the
 * column-concatenated N; each column lands in the segment that holds it, at
 * its offset from the segment start. */
int gq4o_quad_matvec(int M, int K, int N, int gs, int n0, int n1, int n2,
                     const float *A, const uint32_t *Bq, const float *scales,
                     const float *zeros, double *out0, double *out1,
                     double *out2, double *out3, double *S0, double *S1,
                     double *S2, double *S3)
{
    if (!shape_ok(M, K, N, gs) || !A || !Bq || !scales || !zeros) return -1;
    if (!(0 <= n0 && n0 <= n1 && n1 <= n2 && n2 <= N)) return -1;
    const int start[4] = {0, n0, n1, n2};
    const int len[4] = {n0, n1 - n0, n2 - n1, N - n2};
    double *const out[4] = {out0, out1, out2, out3};
    double *const sabs[4] = {S0, S1, S2, S3};
    for (int i = 0; i < 4; ++i)
        if (len[i] > 0 && !out[i]) return -1;

    for (int m = 0; m < M; ++m) {
        for (int col = 0; col < N; ++col) {
            double s_abs = 0.0;
            const double total = dot_f32(K, gs, A + (size_t)m * K, Bq, scales,
                                         zeros, col, &s_abs);
            int seg;
            if (col < n0) seg = 0;
            else if (col < n1) seg = 1;
            else if (col < n2) seg = 2;
            else seg = 3;
            const size_t at = (size_t)m * len[seg] + (size_t)(col - start[seg]);
            out[seg][at] = total;
            if (sabs[seg]) sabs[seg][at] = s_abs;
        }
    }
    return 0;
}

/* RMSNorm prologue (WGSL_NORM_MATVEC_INT4 prologue): x = A_a + A_b as one
 * binary32 addition per element, the mean of x^2 over the K elements of the
 * sum, inv_rms = 1/sqrt(mean + eps), and the normalised activation
 * x * inv_rms * W_norm.  eps is the binary32 value the params carry. */
int gq4o_norm(int M, int K, const float *A_a, const float *A_b,
              const float *W_norm, float eps, float *x, double *a,
              double *inv)
{
    if (M <= 0 || K <= 0 || !A_a || !W_norm || !a) return -1;
    for (int m = 0; m < M; ++m) {
        const float *aa = A_a + (size_t)m * K;
        const float *ab = A_b ? A_b + (size_t)m * K : NULL;
        double sum_sq = 0.0;
        for (int k = 0; k < K; ++k) {
            volatile float xk = ab ? aa[k] + ab[k] : aa[k];
            if (x) x[(size_t)m * K + k] = xk;
            sum_sq += (double)xk * (double)xk;
        }
        const double inv_rms = 1.0 / sqrt(sum_sq / (double)K + (double)eps);
        if (inv) inv[m] = inv_rms;
        for (int k = 0; k < K; ++k) {
            volatile float xk = ab ? aa[k] + ab[k] : aa[k];
            a[(size_t)m * K + k] = (double)xk * inv_rms * (double)W_norm[k];
        }
    }
    return 0;
}

int gq4o_norm_matvec(int M, int K, int N, int gs, const float *A_a,
                     const float *A_b, const float *W_norm, float eps,
                     const uint32_t *Bq, const float *scales,
                     const float *zeros, double *C, double *S,
                     float *residual_out, double *norm_out)
{
    if (!shape_ok(M, K, N, gs) || !A_a || !W_norm || !Bq || !scales ||
        !zeros || !C)
        return -1;
    /* Step 1: the prologue for every lane.  Step 2: the plain matvec on the
     * normalised activations. */
    double *a = norm_out ? norm_out : (double *)malloc(sizeof(double) * (size_t)M * (size_t)K);
    if (!a) return -1;
    int rc = gq4o_norm(M, K, A_a, A_b, W_norm, eps, residual_out, a, NULL);
    for (int m = 0; rc == 0 && m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            double s_abs = 0.0;
            C[(size_t)m * N + n] =
                gq4o_dot(K, gs, a + (size_t)m * K, Bq, scales, zeros, n, &s_abs);
            if (S) S[(size_t)m * N + n] = s_abs;
        }
    }
    if (a != norm_out) free(a);
    return rc;
}

/* silu(t) = t * sigmoid(t) = t / (1 + exp(-t)) (executor declarations,
 * the SwiGLU fusion docs: "silu(gate) * up"). */
static double silu(double t)
{
    return t / (1.0 + exp(-t));
}

int gq4o_gated_matvec(int M, int K, int N, int gs, const float *A,
                      const float *A_b, const float *W_norm, float eps,
                      const uint32_t *Bq_gate, const float *scales_gate,
                      const float *zeros_gate, const uint32_t *Bq_up,
                      const float *scales_up, const float *zeros_up,
                      double *out, double *g, double *u, double *Sg,
                      double *Su, float *residual_out, double *norm_out)
{
    if (!shape_ok(M, K, N, gs) || !A || !Bq_gate || !scales_gate ||
        !zeros_gate || !Bq_up || !scales_up || !zeros_up || !out)
        return -1;
    if (!W_norm && (A_b || residual_out || norm_out)) return -1;

    /* The activation: A itself, or the RMSNorm prologue of A (+ A_b). */
    double *a = norm_out ? norm_out : (double *)malloc(sizeof(double) * (size_t)M * (size_t)K);
    if (!a) return -1;
    int rc = 0;
    if (W_norm) {
        rc = gq4o_norm(M, K, A, A_b, W_norm, eps, residual_out, a, NULL);
    } else {
        for (size_t i = 0; i < (size_t)M * (size_t)K; ++i) a[i] = (double)A[i];
    }
    for (int m = 0; rc == 0 && m < M; ++m) {
        const double *am = a + (size_t)m * K;
        for (int n = 0; n < N; ++n) {
            double sg = 0.0, su = 0.0;
            const double gv = gq4o_dot(K, gs, am, Bq_gate, scales_gate, zeros_gate, n, &sg);
            const double uv = gq4o_dot(K, gs, am, Bq_up, scales_up, zeros_up, n, &su);
            const size_t at = (size_t)m * N + n;
            out[at] = silu(gv) * uv;
            if (g) g[at] = gv;
            if (u) u[at] = uv;
            if (Sg) Sg[at] = sg;
            if (Su) Su[at] = su;
        }
    }
    if (a != norm_out) free(a);
    return rc;
}

/* sigmoid(t) = 1 / (1 + exp(-t)) (the attention SigmoidGate of the
 * GatedMatVecInt4 fusion doc: "attn_out * sigmoid(gate)"). */
static double sigmoid(double t)
{
    return 1.0 / (1.0 + exp(-t));
}

int gq4o_gated_input_matvec(int M, int K, int N, int gs, int kind, const float *X,
                            const float *Gt, const uint32_t *Bq, const float *scales,
                            const float *zeros, double *C, double *S, double *a_out)
{
    if (!shape_ok(M, K, N, gs) || !X || !Gt || !Bq || !scales || !zeros || !C) return -1;
    if (kind != 0 && kind != 1) return -1;
    double *a = a_out ? a_out : (double *)malloc(sizeof(double) * (size_t)M * (size_t)K);
    if (!a) return -1;
    /* The input vector: kind 0, x * sigmoid(g) (GatedMatVecInt4); kind 1,
     * silu(g) * x (SwiGLUGatedMatVecInt4: "silu(gate) * up", x = up). */
    for (size_t i = 0; i < (size_t)M * (size_t)K; ++i) {
        const double x = (double)X[i], g = (double)Gt[i];
        a[i] = kind == 0 ? x * sigmoid(g) : silu(g) * x;
    }
    for (int m = 0; m < M; ++m) {
        const double *am = a + (size_t)m * K;
        for (int n = 0; n < N; ++n) {
            double sabs = 0.0;
            C[(size_t)m * N + n] = gq4o_dot(K, gs, am, Bq, scales, zeros, n, &sabs);
            if (S) S[(size_t)m * N + n] = sabs;
        }
    }
    if (a != a_out) free(a);
    return 0;
}

/* ---- Quantizer and MLX conversion --------------------------------------- */

int gq4o_quantize(int K, int N, int gs, const float *W, uint32_t *Bq,
                  float *scales, float *zeros, int *bad_groups)
{
    if (!shape_ok(1, K, N, gs) || !W || !Bq || !scales || !zeros) return -1;
    const int G = K / gs;
    int bad_count = 0;
    for (size_t i = 0; i < (size_t)N * (size_t)(K / 8); ++i) Bq[i] = 0u;
    for (int n = 0; n < N; ++n) {
        for (int g = 0; g < G; ++g) {
            const float *v = W + (size_t)n * K + (size_t)g * gs;
            const size_t gi = (size_t)n * G + g;
            int bad = 0;
            for (int i = 0; i < gs; ++i)
                if (!isfinite(v[i])) bad = 1;
            volatile float lo = 0.0f, hi = 0.0f, d = 0.0f;
            if (!bad) {
                lo = v[0];
                hi = v[0];
                for (int i = 1; i < gs; ++i) {
                    if (v[i] < lo) lo = v[i];
                    if (v[i] > hi) hi = v[i];
                }
                lo = lo + 0.0f;  /* -0 becomes +0 */
                hi = hi + 0.0f;
                d = hi - lo;
                if (!isfinite(d)) bad = 1;
            }
            if (bad) {
                /* codes stay 0 */
                scales[gi] = NAN;
                zeros[gi] = NAN;
                ++bad_count;
                continue;
            }
            volatile float s = d / 15.0f;
            if (s < FLT_MIN) s = 1.0f;
            volatile float r = 1.0f / s;
            volatile float z = -lo / s;
            for (int i = 0; i < gs; ++i) {
                volatile float diff = v[i] - lo;
                volatile float t = diff * r;
                float qf = rintf(t);
                if (qf < 0.0f) qf = 0.0f;
                if (qf > 15.0f) qf = 15.0f;
                const int k = g * gs + i;
                Bq[(size_t)n * (K / 8) + k / 8] |= (uint32_t)qf << (4 * (k % 8));
            }
            scales[gi] = s;
            zeros[gi] = z;
        }
    }
    if (bad_groups) *bad_groups = bad_count;
    return 0;
}

int gq4o_mlx_dequant_f64(int K, int N, int gs, const uint32_t *packed,
                         const float *mlx_scales, const float *mlx_biases,
                         double *W)
{
    if (!shape_ok(1, K, N, gs) || !packed || !mlx_scales || !mlx_biases || !W) return -1;
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            const size_t g = group_index(K, gs, n, k);
            const double q = (double)gq4o_nibble(packed, K, n, k);
            W[(size_t)n * K + k] = (double)mlx_scales[g] * q + (double)mlx_biases[g];
        }
    }
    return 0;
}

int gq4o_from_mlx(int K, int N, int gs, const uint32_t *packed,
                  const float *mlx_scales, const float *mlx_biases,
                  uint32_t *Bq, float *scales, float *zeros)
{
    if (!shape_ok(1, K, N, gs) || !packed || !mlx_scales || !mlx_biases) return -1;
    if (!Bq || !scales || !zeros) return -1;
    const int G = K / gs;
    for (size_t i = 0; i < (size_t)N * (size_t)(K / 8); ++i) Bq[i] = packed[i];
    for (size_t gi = 0; gi < (size_t)N * (size_t)G; ++gi) {
        const float s = mlx_scales[gi], b = mlx_biases[gi];
        volatile float z = -b / s;
        if (s == 0.0f || (isinf(z) && isfinite(b))) {
            /* w = b for every code: codes 1, scale b, zero 0 */
            const size_t w0 = gi * (size_t)(gs / 8);
            for (int j = 0; j < gs / 8; ++j) Bq[w0 + j] = 0x11111111u;
            scales[gi] = b;
            zeros[gi] = 0.0f;
        } else {
            scales[gi] = s;
            zeros[gi] = z;
        }
    }
    return 0;
}

/* ---- Embedding gather --------------------------------------------------- */

int gq4o_embedding(int T, int K, int V, int gs, const int32_t *ids,
                   const uint32_t *Bq, const float *scales, const float *zeros,
                   float *out, int *bad_ids)
{
    if (T < 0 || !shape_ok(1, K, V, gs) || !Bq || !scales || !zeros) return -1;
    if (T > 0 && (!ids || !out)) return -1;
    int bad = 0;
    for (int t = 0; t < T; ++t) {
        const int32_t v = ids[t];
        float *row = out + (size_t)t * K;
        if (v < 0 || v >= V) {
            for (int k = 0; k < K; ++k) row[k] = NAN;
            ++bad;
            continue;
        }
        for (int k = 0; k < K; ++k) {
            const size_t g = group_index(K, gs, v, k);
            volatile float d = (float)gq4o_nibble(Bq, K, v, k) - zeros[g];
            volatile float w = d * scales[g];
            row[k] = w;
        }
    }
    if (bad_ids) *bad_ids = bad;
    return 0;
}

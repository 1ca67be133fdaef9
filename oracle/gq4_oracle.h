/*
 * gq4_oracle.h -- plain CPU oracle for the int4 group-quantized matvec family.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a slow, obviously-correct restatement in
 * C99 of what the int4 weight-only group-quantized matrix-vector product
 * computes, accumulated in double precision.  It exists to check the CUDA
 * library against.  Only the test suite, the smoke check and the CPU baseline
 * leg of the benchmark may load it; the product path never does.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Source of the definitions (gerbil 1.12.0 -> 1.13.0 diffs):
 *   - weight layout: gpu bundle, Gepard graph builder `addLinearOp` (q is
 *     ceil(K*N/8) u32 words, scales/zeros ceil(K*N/gs) f32 each) and the
 *     executor declarations, `fuseMambaFrontDecodeEntries` doc ("stored
 *     column-major, one column contiguous");
 *   - nibble order, group index and dequant rule w = (q - zero) * scale:
 *     moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 main loop;
 *   - quad routing at n0/n1/n2: WGSL_QUAD_MATVEC_INT4 epilogue and
 *     QUAD_MATVEC_INT4_SPEC params {K, N, group_size, n0, n1, n2};
 *   - RMSNorm prologue: WGSL_NORM_MATVEC_INT4 prologue and
 *     NORM_MATVEC_INT4_SPEC (eps passed as f32 bits, default 1e-6);
 *   - SiLU-gated gate/up: executor declarations, fuseSwiGLUDecodeEntries doc
 *     ("silu(gate) * up") and the NormSwiGLUMatVec fusion doc.
 *
 * Conventions: M lanes, K inputs, N output columns, group size gs, G = K/gs.
 * A is f32 [M][K]; Bq is u32 [N][K/8] (column n owns words n*K/8 .. n*K/8+K/8-1,
 * element k is nibble k%8 of word k/8, low nibble first); scales and zeros are
 * f32 [N][G].  Results are double.  For every result the oracle also returns
 * S = sum_k |a_k * w(n,k)|, the scale of the parity tolerance.
 *
 * Every function returns 0 on success and -1 on an invalid argument (the
 * shape rules are the ones the layout needs: K > 0 with K % 8 == 0, gs > 0
 * with K % gs == 0, N > 0, M > 0).
 */
#ifndef GQ4_ORACLE_H
#define GQ4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* q(n,k): the 4-bit code of element k of column n. */
int gq4o_nibble(const uint32_t *Bq, int K, int n, int k);

/* Unpack every code: q[n*K + k] = q(n,k). */
int gq4o_unpack(int K, int N, const uint32_t *Bq, uint8_t *q);

/* Inverse of gq4o_unpack: pack codes q[n*K + k] (each 0..15) into Bq. */
int gq4o_pack(int K, int N, const uint8_t *q, uint32_t *Bq);

/* w(n,k) = (q - zero) * scale, exactly (double). W is [N][K]. */
int gq4o_dequant_f64(int K, int N, int gs, const uint32_t *Bq,
                     const float *scales, const float *zeros, double *W);

/* The same rule evaluated in binary32 with one rounding per operation:
 * t = fl32((float)q - zero), w = fl32(t * scale).  W is [N][K]. */
int gq4o_dequant_f32(int K, int N, int gs, const uint32_t *Bq,
                     const float *scales, const float *zeros, float *W);

/* One output: sum_k a[k] * w(n,k) in increasing k (double); *S gets the
 * absolute sum.  a is a double vector of length K. */
double gq4o_dot(int K, int gs, const double *a, const uint32_t *Bq,
                const float *scales, const float *zeros, int n, double *S);

/* C[m][n] = sum_k A[m][k] * w(n,k).  C and S are [M][N] (S may be NULL). */
int gq4o_matvec(int M, int K, int N, int gs, const float *A,
                const uint32_t *Bq, const float *scales, const float *zeros,
                double *C, double *S);

/* The same for a subset of columns and double activations a [M][K]:
 * C[m][j] = dot(a[m], cols[j]).  C and S are [M][ncols] (S may be NULL). */
int gq4o_matvec_cols(int M, int K, int gs, const double *a,
                     const uint32_t *Bq, const float *scales,
                     const float *zeros, int ncols, const int *cols,
                     double *C, double *S);

/* Quad-output matvec: the unsplit matvec over N columns, each column routed
 * to out0 (col < n0), out1 (n0 <= col < n1), out2 (n1 <= col < n2) or out3
 * (col >= n2) at offset col - (start of its segment).  out_i is
 * [M][len_i] with len = {n0, n1-n0, n2-n1, N-n2}; an empty segment's
 * pointers may be NULL.  S_i (nullable) mirror out_i. */
int gq4o_quad_matvec(int M, int K, int N, int gs, int n0, int n1, int n2,
                     const float *A, const uint32_t *Bq, const float *scales,
                     const float *zeros, double *out0, double *out1,
                     double *out2, double *out3, double *S0, double *S1,
                     double *S2, double *S3);

/* RMSNorm prologue on x = A_a + A_b (A_b may be NULL: x = A_a):
 *   x[k]   = A_a[k] + A_b[k]           (one binary32 addition)
 *   inv    = 1 / sqrt(sum_k x[k]^2 / K + eps)    (double)
 *   a[k]   = x[k] * inv * W_norm[k]               (double)
 * x (nullable) is [M][K] float, a is [M][K] double, inv (nullable) is [M]. */
int gq4o_norm(int M, int K, const float *A_a, const float *A_b,
              const float *W_norm, float eps, float *x, double *a,
              double *inv);

/* Norm-prologue matvec: C[m][n] = dot(a[m], n) with a from gq4o_norm.
 * residual_out (= x, float) and norm_out (= a, double) are nullable. */
int gq4o_norm_matvec(int M, int K, int N, int gs, const float *A_a,
                     const float *A_b, const float *W_norm, float eps,
                     const uint32_t *Bq, const float *scales,
                     const float *zeros, double *C, double *S,
                     float *residual_out, double *norm_out);

/* SiLU-gated gate/up matvec: g = dot(a, Wg col n), u = dot(a, Wu col n),
 * out = silu(g) * u with silu(t) = t / (1 + exp(-t)).  a = A (W_norm NULL)
 * or the RMSNorm prologue of A (+ A_b) with W_norm and eps.  g, u, Sg, Su,
 * residual_out, norm_out are nullable; all but the last two are [M][N]. */
int gq4o_gated_matvec(int M, int K, int N, int gs, const float *A,
                      const float *A_b, const float *W_norm, float eps,
                      const uint32_t *Bq_gate, const float *scales_gate,
                      const float *zeros_gate, const uint32_t *Bq_up,
                      const float *scales_up, const float *zeros_up,
                      double *out, double *g, double *u, double *Sg,
                      double *Su, float *residual_out, double *norm_out);

/* Gated-input matvec: the input vector is built from two [M][K] vectors and
 * then multiplied like gq4o_matvec.  kind 0: a = X * sigmoid(G) (the
 * attention SigmoidGate fused into o_proj, GatedMatVecInt4 fusion doc);
 * kind 1: a = silu(G) * X (a standalone SwiGLU "silu(gate) * up" fused into
 * the consuming projection, SwiGLUGatedMatVecInt4 fusion doc; X = up).
 * C, S as gq4o_matvec; a_out (optional) receives a [M][K]. */
int gq4o_gated_input_matvec(int M, int K, int N, int gs, int kind, const float *X,
                            const float *G, const uint32_t *Bq, const float *scales,
                            const float *zeros, double *C, double *S, double *a_out);

/* ---- The step before the path: producing the format ----------------------
 *
 * Group-wise int4 quantizer (the backbone's weight-only INT4 of the gpu
 * bundle's loader, quantizeInt4 / quantizeBackboneInt4, whose body the pages
 * do not show).  Reading: per group of gs consecutive inputs of a column, a
 * min/max asymmetric affine map onto the 16 codes with a float zero point,
 * every step one binary32 operation (the precision in which the codes are
 * decided):
 *   lo = min v, hi = max v             (+0.0 added: no negative zero)
 *   s  = fl(fl(hi - lo) / 15)          s < FLT_MIN (a range below 15 normal
 *                                      steps, e.g. a constant group): s = 1
 *   z  = fl(-lo / s)
 *   q  = clamp(rint(fl(fl(v - lo) * fl(1 / s))), 0, 15)   (ties to even)
 * so that (q - z) * s is the nearest of the 16 levels lo + j*s.  A group with
 * a non-finite value, or whose range hi - lo overflows, gets codes 0 and a
 * NaN scale and zero.  W is f32 [N][K] (column n's K weights contiguous:
 * W[n][k] multiplies input k for output n).  *bad_groups (nullable) receives
 * the number of such groups. */
int gq4o_quantize(int K, int N, int gs, const float *W, uint32_t *Bq,
                  float *scales, float *zeros, int *bad_groups);

/* MLX affine int4 (gpu bundle 1.0.0, dequantizeMLXProjection): the same
 * words (8 codes per u32, low nibble first, rows = output columns, groups of
 * gs along the row) with w = scale * q + bias.  Dequantized in double:
 * W[n][k] = (double)scale * q + (double)bias.  W is [N][K]. */
int gq4o_mlx_dequant_f64(int K, int N, int gs, const uint32_t *packed,
                         const float *mlx_scales, const float *mlx_biases,
                         double *W);

/* MLX (scale, bias) to this format's (scale, zero): zero = fl(-bias / scale)
 * in binary32, codes unchanged, so (q - zero) * scale = scale * q + bias.
 * A group that has no such zero (scale 0, or -bias/scale overflowing while
 * bias is finite; then w = bias for every code, to within bias's own
 * rounding) is rewritten exactly: all its codes 1, scale = bias, zero = 0.
 * Bq may be packed (in place). */
int gq4o_from_mlx(int K, int N, int gs, const uint32_t *packed,
                  const float *mlx_scales, const float *mlx_biases,
                  uint32_t *Bq, float *scales, float *zeros);

/* Int4 embedding gather (the decode step's first dispatch, EmbeddingInt4, and
 * the per-layer-embedding row gather of the gpu bundle's executor, which
 * dequantizes only the rows of the step's token ids from a table
 * {packed, scales, zeros, width, groupSize}).  The table is V rows of width
 * K in this format (row v = "column" v: K/8 words, K/gs groups).  For each of
 * T token ids: out[t][k] = fl(fl(q(ids[t], k) - zero) * scale), the binary32
 * dequant of gq4o_dequant_f32.  An id outside [0, V) gives a row of NaN and
 * is counted in *bad_ids (nullable).  out is f32 [T][K]. */
int gq4o_embedding(int T, int K, int V, int gs, const int32_t *ids,
                   const uint32_t *Bq, const float *scales, const float *zeros,
                   float *out, int *bad_ids);

#ifdef __cplusplus
}
#endif

#endif /* GQ4_ORACLE_H */

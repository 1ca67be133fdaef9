/*
 * gq4.h -- C ABI of libgq4: the int4 weight-only group-quantized
 * matrix-vector product used in LLM token decode, with its fused variants,
 * for NVIDIA GB300 (sm_103a).
 *
 * Source of the operations (gerbil 1.12.0 -> 1.13.0 bundle diffs):
 *   - format and dequant rule: moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4
 *     main loop; gpu bundle, Gepard graph builder `addLinearOp` (tensors
 *     `.q` u32, `.scales` / `.zeros` f32); executor declarations,
 *     `fuseMambaFrontDecodeEntries` doc (weights column-major, one column
 *     contiguous);
 *   - quad routing: WGSL_QUAD_MATVEC_INT4 epilogue and QUAD_MATVEC_INT4_SPEC
 *     (bindings A, B_q, scales, zeros, out0..out3, params {K, N, group_size,
 *     n0, n1, n2});
 *   - RMSNorm prologue: WGSL_NORM_MATVEC_INT4 and NORM_MATVEC_INT4_SPEC
 *     (bindings A_a, A_b, W_norm, B_q, scales, zeros, C, residual_out,
 *     norm_out, params {K, N, group_size, eps});
 *   - SiLU-gated gate/up: executor declarations, fuseSwiGLUDecodeEntries and
 *     fuseNormSwiGLUDecodeEntries docs (silu(gate) * up, optional residual +
 *     RMSNorm prologue);
 *   - batched lanes: executor declarations, buildBatchEntries doc (lanes run
 *     the same weights and never interact);
 *   - dual projection: executor declarations, fuseDualMatVecDecodeEntries doc
 *     (two projections sharing the input and K/N, numerics of two matvecs);
 *   - gated inputs: executor declarations, fuseGatedOProjDecodeEntries doc
 *     (attn_out * sigmoid(gate) into o_proj) and
 *     fuseSwiGLUGatedProjDecodeEntries doc (silu(gate) * up into the
 *     consuming projection);
 *   - producing the format: the gpu bundle's loader (the backbone's linears
 *     quantized weight-only, group-wise to INT4 by quantizeInt4 /
 *     quantizeBackboneInt4, body not shown) and the gpu bundle 1.0.0
 *     dequantizeMLXProjection (MLX affine int4, w = scale * q + bias);
 *   - prefill GEMM: executor declarations, dispatchEntries (prefill as tiled
 *     matrix multiplies over the same weights);
 *   - embedding gather: executor declarations, EmbeddingInt4 (the decode
 *     step's first kernel) and setPleSource / streamPleRows (an int4 table
 *     {packed, scales, zeros, width, groupSize} of which only the rows of the
 *     step's token ids are dequantized).
 *
 * ---------------------------------------------------------------------------
 * Weight format (one int4 matrix of K inputs and N output columns, group size
 * gs, G = K / gs groups per column):
 *   Bq      u32 [N][K/8]   column n owns words n*K/8 .. n*K/8 + K/8 - 1;
 *                          element k of column n is bits 4*(k%8) .. 4*(k%8)+3
 *                          of word k/8 (low nibble first), a code q in 0..15.
 *   scales  f32 [N][G]     one per (column, group of gs consecutive k).
 *   zeros   f32 [N][G]     one per (column, group); need not be an integer.
 *   w(n,k) = (q(n,k) - zeros[n][k/gs]) * scales[n][k/gs].
 * Activations A are f32 [M][K] (lane-major), outputs f32 [M][len].
 * C[m][n] = sum_k A[m][k] * w(n,k).
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer owned by the caller; the caller keeps
 *     the buffers alive until the stream has passed the call.  The library
 *     allocates no memory and never synchronizes on the call path; its only
 *     state is its sticky device-side error bits (gq4_device_error) and a
 *     per-device cache of launch geometry.
 *   - All checks run on the host before anything is enqueued.  A status other
 *     than GQ4_OK means nothing was enqueued on the stream.  GQ4_ERR_CUDA
 *     means a launch was rejected by the CUDA runtime (cudaGetLastError);
 *     errors raised later by the kernel surface on the stream as usual.
 *   - Shape rules: 1 <= M <= GQ4_MAX_LANES, K > 0, N > 0,
 *     group_size % 32 == 0, K % group_size == 0.  (Every element group then
 *     holds whole 32-code / 16-byte chunks, the unit of the 128-bit loads.)
 *   - Alignment: Bq, A and every [M][K] vector 16-byte aligned; scales, zeros
 *     and outputs 4-byte aligned.  Otherwise GQ4_ERR_MISALIGNED.
 *   - Outputs must not overlap each other or any input (GQ4_ERR_ALIAS).
 *   - Launches are asynchronous on `stream` (0 = the legacy default stream).
 *     Stream order holds for activations, norm inputs and outputs.  One
 *     exception for weights: calls with M <= 4 or 16 <= M <= 32 may be
 *     launched with programmatic dependent launch, so such a call may start reading
 *     its Bq, scales and zeros before the kernel just before it on the same
 *     stream has completed: while it runs, if it is one of these matvecs
 *     (which signal early), else once its blocks have exited.  Hence:
 *       - the weights of a call must not be outputs of the matvec call
 *         immediately preceding it;
 *       - any other kernel that writes a call's weights and immediately
 *         precedes it on the stream must make those stores visible GPU-wide
 *         before its blocks exit (every writing thread executes
 *         __threadfence() after its last store, as gq4_quantize and
 *         gq4_from_mlx do), or the caller puts a non-kernel operation
 *         (an event wait, a copy) or a host synchronisation in between.
 *   - Results are deterministic: the same inputs give the same bits.
 *   - A NaN or infinite activation makes every output whose dot product uses
 *     it non-finite (NaN at M = 1 and on the 2..4-lane kernel below).
 *   - Arithmetic: with 2 <= M <= 4 lanes, a group size that is a power-of-
 *     two multiple of 128 and K a multiple of 128 that splits into at most
 *     four chunks of whole groups, each at most 32 groups and 32 blocks of
 *     128 codes (one chunk up to K = 4096; e.g. K = 11008 at group 128 in
 *     four; the chunks' f32 sums are added in chunk order), each 128-code
 *     block of a lane's activations is held
 *     as 22-bit fixed point with a power-of-two scale (each value within
 *     2^-22 of the block's largest magnitude), split into two pieces exact
 *     in fp16, and the tensor core's warp-level MMA sums the products
 *     exactly (every partial sum an integer times 2^-24 below 2^24 of them);
 *     the bound below holds unless a block holds an activation some 2^10
 *     times larger than the ones that carry the result.  Other 2 <= M <= 15
 *     calls: every product and sum is f32
 *     (|error| <= 1e-4 * sum_k |a_k w_k| + 1e-6 against the exact dot
 *     product).  With M = 1 each 64-code group of activations is held as
 *     24-bit fixed point with a power-of-two scale (each value within
 *     2^-22 of the group's largest magnitude) and the products are summed
 *     exactly in integers: the same bound holds unless a group holds an
 *     activation some 2^12 times larger than the ones that carry the
 *     result (a huge activation on a near-zero weight).  With
 *     16 <= M <= 32 lanes on sm_103 the weights and the activations are
 *     rounded to bf16 and multiplied on the tensor core with f32
 *     accumulation (|error| <= 2e-2 * sum_k |a_k w_k| + 1e-6); the norm
 *     prologue's side outputs stay f32.
 * ---------------------------------------------------------------------------
 */
#ifndef GQ4_H
#define GQ4_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQ4_MAX_LANES 32
#define GQ4_MAX_GEMM_ROWS (1 << 20)

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define GQ4_API __attribute__((visibility("default")))
#else
#define GQ4_API
#endif

typedef enum gq4_status {
    GQ4_OK = 0,
    GQ4_ERR_INVALID_ARG = 1, /* a shape rule or a required pointer is violated */
    GQ4_ERR_UNSUPPORTED = 2, /* valid request this build does not implement */
    GQ4_ERR_ALIAS = 3,       /* an output overlaps another output or an input */
    GQ4_ERR_CUDA = 4,        /* the CUDA runtime rejected a launch */
    GQ4_ERR_MISALIGNED = 5   /* a pointer breaks its alignment rule */
} gq4_status;

/* Optional residual + RMSNorm prologue (WGSL_NORM_MATVEC_INT4 prologue):
 *   x[m][k]   = A[m][k] + A_b[m][k]                (A_b == NULL: x = A)
 *   inv_rms   = 1 / sqrt(sum_k x[m][k]^2 / K + eps)
 *   a[m][k]   = x[m][k] * inv_rms * W_norm[k]      (the matvec activation)
 * residual_out[m][k] = x (bit-exact f32 sum) and norm_out[m][k] = a are
 * written for every lane when non-NULL. */
typedef struct gq4_norm {
    const float *A_b;     /* [M][K] second addend, or NULL */
    const float *W_norm;  /* [K] gain, required */
    float eps;            /* e.g. 1e-6f; must be >= 0 */
    float *residual_out;  /* [M][K] or NULL */
    float *norm_out;      /* [M][K] or NULL */
} gq4_norm;

/* Plain matvec (the base decode MatMulInt4): C [M][N]. */
GQ4_API gq4_status gq4_matvec(int M, int K, int N, int group_size,
                      const float *A, const uint32_t *Bq,
                      const float *scales, const float *zeros,
                      float *C, cudaStream_t stream);

/* Quad-output matvec over a column-concatenated weight matrix (the byte
 * append of up to four projections sharing A, K and group_size).  Column
 * col goes to out0[m][col] (col < n0), out1[m][col-n0] (n0 <= col < n1),
 * out2[m][col-n1] (n1 <= col < n2) or out3[m][col-n2] (col >= n2).
 * Requires 0 <= n0 <= n1 <= n2 <= N; out_i is [M][len_i] with
 * len = {n0, n1-n0, n2-n1, N-n2} and may be NULL exactly when len_i == 0.
 * Each column's value is bit-identical to gq4_matvec on the same weights. */
GQ4_API gq4_status gq4_quad_matvec(int M, int K, int N, int group_size,
                           int n0, int n1, int n2,
                           const float *A, const uint32_t *Bq,
                           const float *scales, const float *zeros,
                           float *out0, float *out1, float *out2, float *out3,
                           cudaStream_t stream);

/* Norm-prologue matvec: C [M][N] = matvec of the RMSNorm prologue of A
 * (+ norm->A_b).  norm must be non-NULL with W_norm set. */
GQ4_API gq4_status gq4_norm_matvec(int M, int K, int N, int group_size,
                           const gq4_norm *norm,
                           const float *A, const uint32_t *Bq,
                           const float *scales, const float *zeros,
                           float *C, cudaStream_t stream);

/* SiLU-gated gate/up matvec: out[m][n] = silu(g) * u with
 * g = a . w_gate(n, .), u = a . w_up(n, .), silu(t) = t / (1 + exp(-t)).
 * Both matrices are K x N with the same group_size.  a = A, or the RMSNorm
 * prologue of A when norm != NULL (applied once, shared by both). */
GQ4_API gq4_status gq4_gated_matvec(int M, int K, int N, int group_size,
                            const gq4_norm *norm, const float *A,
                            const uint32_t *Bq_gate, const float *scales_gate,
                            const float *zeros_gate,
                            const uint32_t *Bq_up, const float *scales_up,
                            const float *zeros_up,
                            float *out, cudaStream_t stream);

/* Dual projection (DualMatVecInt4): C0 = A . W0 and C1 = A . W1, two K x N
 * matrices with the same group_size over the same input, in one launch.
 * Each output equals gq4_matvec of its matrix within the fp32 tolerance; for
 * M = 1 bit for bit (the same per-column arithmetic).  C0 and C1 are [M][N]
 * and must not overlap each other or any input. */
GQ4_API gq4_status gq4_dual_matvec(int M, int K, int N, int group_size, const float *A,
                                   const uint32_t *Bq0, const float *scales0, const float *zeros0,
                                   const uint32_t *Bq1, const float *scales1, const float *zeros1,
                                   float *C0, float *C1, cudaStream_t stream);

/* Sigmoid-gated input (GatedMatVecInt4): C = a . W with
 * a[m][k] = X[m][k] * sigmoid(G[m][k]), sigmoid(t) = 1 / (1 + exp(-t))
 * (X = the attention output, G = its gate).  X and G are [M][K], 16-byte
 * aligned, read only; the gated vector is formed in the kernel (f32). */
GQ4_API gq4_status gq4_sigmoid_gated_matvec(int M, int K, int N, int group_size, const float *X,
                                            const float *G, const uint32_t *Bq,
                                            const float *scales, const float *zeros, float *C,
                                            cudaStream_t stream);

/* SwiGLU-gated input (SwiGLUGatedMatVecInt4): C = a . W with
 * a[m][k] = silu(G[m][k]) * X[m][k], silu(t) = t / (1 + exp(-t)) (G = the
 * gate, X = the up vector).  Layout and rules as gq4_sigmoid_gated_matvec. */
GQ4_API gq4_status gq4_swiglu_gated_matvec(int M, int K, int N, int group_size, const float *X,
                                           const float *G, const uint32_t *Bq,
                                           const float *scales, const float *zeros, float *C,
                                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Prefill and wide batches: the int4 GEMM.
 *
 * On the pages, prompt processing (prefill) multiplies all the prompt's rows
 * by the same int4 weights in tiled matrix-multiply kernels (the executor's
 * dispatchEntries).  gq4_gemm
 * computes C[m][n] = sum_k A[m][k] * w(n,k) for any 1 <= M <=
 * GQ4_MAX_GEMM_ROWS rows, with the weight format, shape rules, alignment,
 * aliasing and stream rules of gq4_matvec.  Every row is computed on the
 * bf16 tensor cores with f32 accumulation (|error| <= 2e-2 * sum_k |a_k w_k|
 * + 1e-6).  With more than 32 rows and a workspace of at least
 * gq4_gemm_workspace_bytes(M, K) bytes (device memory, 256-byte aligned, not
 * overlapping any argument; its contents on entry do not matter and are
 * overwritten with a bf16 copy of A) the rows run as tiles of a dedicated
 * GEMM kernel that dequantizes each weight tile once per 64..256 rows.
 * Otherwise (M <= 32, workspace NULL or too small) the rows run in chunks
 * of up to 32 on the decode tensor-core kernel (fewer than 16 padded to 16).
 * Where neither tensor-core kernel can take the call (scales or zeros not
 * 16-byte aligned, a device other than sm_103) the chunks run on the f32
 * kernels, within the same bound.
 * ------------------------------------------------------------------------ */
GQ4_API size_t gq4_gemm_workspace_bytes(int M, int K);

GQ4_API gq4_status gq4_gemm(int M, int K, int N, int group_size, const float *A,
                            const uint32_t *Bq, const float *scales, const float *zeros,
                            float *C, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Producing the format (the step before the matvec).
 * ------------------------------------------------------------------------ */

/* Group-wise int4 quantizer.  W is f32 [N][K], column n's K weights
 * contiguous (W[n][k] multiplies input k for output n: one row of a
 * PyTorch or MLX Linear weight), 16-byte aligned.  Writes Bq, scales and
 * zeros in the format above (Bq 16-byte aligned, scales and zeros 4-byte),
 * none overlapping W or each other.  Per group of group_size consecutive
 * inputs of a column, a min/max asymmetric map onto the 16 codes with a
 * float zero point, every step one binary32 operation, ties to even:
 *   lo, hi = min, max of the group (+0.0 added: no negative zero)
 *   scale  = fl(fl(hi - lo) / 15); 1 when that is below FLT_MIN (a constant
 *            group, or a range under 15 normal steps)
 *   zero   = fl(-lo / scale)
 *   q      = clamp(rint(fl(fl(v - lo) * fl(1 / scale))), 0, 15)
 * The dequantized (q - zero) * scale is the nearest of the group's 16
 * levels, within half a step of v.  A group holding a NaN or an infinity,
 * or whose range hi - lo overflows, gets codes 0 and a NaN scale and zero
 * and sets device error bit 3.  Shape rules as above (no M). */
GQ4_API gq4_status gq4_quantize(int K, int N, int group_size, const float *W, uint32_t *Bq,
                                float *scales, float *zeros, cudaStream_t stream);

/* MLX affine int4 to this format.  packed is the MLX weight, u32 [N][K/8]
 * (rows = output columns, 8 codes per word, low nibble first: the same words
 * as Bq); mlx_scales and mlx_biases are f32 [N][K/group_size], and the MLX
 * weight is w = scale * q + bias.  Writes Bq, scales, zeros with
 * zero = fl(-bias / scale) and codes and scale copied, so that
 * (q - zero) * scale = scale * q + bias up to the one rounding of zero
 * (|error| <= 2^-24 |bias|).  A group without such a zero (scale 0, or
 * -bias / scale overflowing with a finite bias, where w rounds to bias for
 * every code) is written as codes 1, scale = bias, zero 0: exactly w = bias.
 * Non-finite scales or biases propagate.  Bq may be packed itself (in place:
 * only rewritten groups are stored); otherwise no output may overlap an
 * input or another output.  packed and Bq 16-byte aligned, the rest 4-byte. */
GQ4_API gq4_status gq4_from_mlx(int K, int N, int group_size, const uint32_t *packed,
                                const float *mlx_scales, const float *mlx_biases, uint32_t *Bq,
                                float *scales, float *zeros, cudaStream_t stream);

/* Int4 embedding gather.  The table is V rows of width K in the format above
 * (row v is "column" v: Bq u32 [V][K/8], scales and zeros f32 [V][K/gs]);
 * ids is int32 [T] on the device; out is f32 [T][K]:
 *   out[t][k] = fl(fl(q(ids[t], k) - zeros[ids[t]][k/gs]) * scales[...])
 * (one binary32 rounding per operation).  An id outside [0, V) gives a row
 * of NaN and sets device error bit 4; its table row is not read.  T = 0 is
 * a no-op.  Shape rules as above with N = V; out 16-byte aligned, ids 4-byte;
 * out must not overlap any input. */
GQ4_API gq4_status gq4_embedding(int T, int K, int V, int group_size, const int32_t *ids,
                                 const uint32_t *Bq, const float *scales, const float *zeros,
                                 float *out, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * One-lane call sequences (decode of a whole layer stack in one launch).
 *
 * The pages run a decode step as a list of dispatches over the same kernels
 * (the gerbil executor's decode entries: per layer the quad QKV matvec, the
 * output projection, the SiLU-gated gate/up with its norm prologue and the
 * down projection).  gq4_run_sequence runs such a list of one-lane (M = 1)
 * calls, in order, with the semantics of issuing them one by one: call i+1
 * may read what calls 0..i wrote.  It is one persistent launch: while the
 * lanes of call i finish, the weights of call i+1 are already streaming in.
 * ------------------------------------------------------------------------ */
typedef enum gq4_op {
    GQ4_OP_MATVEC = 0,   /* gq4_matvec:       out[0] = C                        */
    GQ4_OP_QUAD = 1,     /* gq4_quad_matvec:  out[0..3], split points n0..n2    */
    GQ4_OP_NORM = 2,     /* gq4_norm_matvec:  out[0] = C, norm required          */
    GQ4_OP_GATED = 3     /* gq4_gated_matvec: out[0], gate = [0], up = [1], norm optional */
} gq4_op;

typedef struct gq4_call {
    int op;                    /* gq4_op */
    int K, N, group_size;
    int n0, n1, n2;            /* GQ4_OP_QUAD only */
    const float *A;            /* [K] */
    const uint32_t *Bq[2];     /* [1], scales[1], zeros[1]: GQ4_OP_GATED's up matrix */
    const float *scales[2];
    const float *zeros[2];
    float *out[4];
    int has_norm;              /* GQ4_OP_NORM: must be 1; GQ4_OP_GATED: optional */
    gq4_norm norm;
} gq4_call;

/* Bytes of device workspace gq4_run_sequence needs (a grid barrier). */
GQ4_API size_t gq4_sequence_workspace_bytes(void);

/* Run n_calls one-lane calls in order on `stream`.  Each call is validated
 * as its single entry point would validate it (M = 1); outputs of one call
 * must not overlap that call's inputs, but later calls may read them.
 * `workspace` is device memory of at least gq4_sequence_workspace_bytes(),
 * 16-byte aligned, that no call touches, zero-filled by the caller before
 * its first use; a completed launch leaves it ready for the next sequence on
 * the same stream (its arrival counter back at zero).
 * Sequences in flight at the same time (other streams) need distinct
 * workspaces.  After a call fails with a device error (gq4_device_error bit
 * 2) the workspace must be zero-filled again.  The launch is cooperative
 * (one CTA per SM, all resident).  Long sequences run as several launches
 * of up to 128 calls each.  A sequence the persistent kernel cannot take
 * (scale or zero rows not 16-byte aligned, shapes whose ring entries do not
 * fit, no room for one CTA per SM) runs as individual launches instead,
 * with the same results. */
GQ4_API gq4_status gq4_run_sequence(const gq4_call *calls, int n_calls, void *workspace,
                                    cudaStream_t stream);

/* How gq4_run_sequence and gq4_run_sequence_static would run `calls`
 * (no counterpart on the pages: it reports the library's own plan).
 * *launches receives the number of persistent launches the sequence takes
 * (one per 128 calls), or 0 when it would run as individual launches of the
 * single-call kernels.  The calls are validated as gq4_run_sequence
 * validates them (the workspace aside); the same statuses are returned and
 * nothing is enqueued.  Host only: reads the current device's attributes. */
GQ4_API gq4_status gq4_sequence_launches(const gq4_call *calls, int n_calls, int *launches);

/* Allocation-free form of gq4_run_sequence, for callers that cannot
 * allocate device memory.  The pages have no counterpart to it: it changes
 * only where the launch's scratch lives.  Same calls, validation, semantics
 * and results as gq4_run_sequence; the grid barrier's counters
 * (gq4_sequence_workspace_bytes() bytes) live in a fixed 256-byte array of
 * this library on the current device instead of a caller workspace.  A
 * sequence whose scratch would exceed that array is rejected with
 * GQ4_ERR_INVALID_ARG before anything is enqueued.  Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library routine; the array's
 * address is looked up once per device.  The counters must start at zero:
 * once every call has passed validation, a call that runs as the persistent
 * launch enqueues a cudaMemsetAsync of them on `stream` right before that
 * launch (a rejected call enqueues nothing; a sequence that runs as
 * individual launches does not touch the array).  All such calls on one
 * device share the array, so calls that overlap on the GPU (other streams,
 * other host threads) race: the caller must order them. */
GQ4_API gq4_status gq4_run_sequence_static(const gq4_call *calls, int n_calls, cudaStream_t stream);

/* Integer unpack test kernel: q[n*K + k] = q(n,k) as u8 [N][K].
 * Uses the same in-register extraction as the matvec kernels.
 * Requires K % 32 == 0. */
GQ4_API gq4_status gq4_unpack(int K, int N, const uint32_t *Bq, uint8_t *q,
                      cudaStream_t stream);

/* Dequant test kernel: W[n*K + k] = fl32(fl32(q - zero) * scale) as f32
 * [N][K], one rounding per operation, through the same extraction as the
 * matvec kernels. */
GQ4_API gq4_status gq4_dequant(int K, int N, int group_size, const uint32_t *Bq,
                       const float *scales, const float *zeros, float *W,
                       cudaStream_t stream);

/* The library's sticky device-side error bits on the current device.  Bit 0
 * is set when the one-lane kernel gave up waiting for one of its own bulk
 * copies, bit 1 when the tensor-core kernel gave up waiting for a copy, an
 * MMA or a peer CTA of its cluster, bit 2 when a call sequence gave up
 * waiting for a copy or for the other CTAs at a call boundary (every wait
 * inside the kernels is bounded in time, so a broken copy cannot hang the
 * GPU; the outputs of that call are then invalid), bit 3 when gq4_quantize
 * met a group with a non-finite value or range, bit 4 when gq4_embedding met
 * an id outside its table, bit 5 when the 2..4-lane kernel gave up waiting
 * for a copy, its scale scratch or its warps' partial sums; bit 1 also
 * covers the GEMM kernel of gq4_gemm.  Copies the word to
 * *bits (synchronous, device-wide) and clears it when clear != 0.  Not for
 * the hot path: a diagnostic to call after a suspicious result. */
GQ4_API gq4_status gq4_device_error(unsigned int *bits, int clear);

/* Static description of a status code. */
GQ4_API const char *gq4_status_string(gq4_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
GQ4_API int gq4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQ4_H */

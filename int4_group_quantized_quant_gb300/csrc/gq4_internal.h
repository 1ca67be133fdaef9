// gq4_internal.h -- host-side interface between the C ABI and the launchers.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "gq4.h"

namespace gq4 {

enum Epilogue : int {
    kEpiStore = 0,  // C[m][col]
    kEpiQuad = 1,   // route col to out0..out3 at the split points
    kEpiGated = 2,  // out[m][col] = silu(gate) * up
    kEpiDual = 3,   // two matrices, one input: out0[m][col], out1[m][col]
};

// How the activation vector is built (kernel template parameter).
enum Prologue : int {
    kProNone = 0,     // a = A
    kProNorm = 1,     // a = RMSNorm(A + A_b) * W_norm
    kProSigmoid = 2,  // a = A * sigmoid(G)
    kProSwiglu = 3,   // a = silu(G) * A
};

// Gated-input kinds of a call (Call::gate_kind).
enum GateKind : int {
    kGateNone = 0,
    kGateSigmoid = 1,
    kGateSwiglu = 2,
};

// One validated call, as the launchers see it.  At most one of norm and
// gate_kind is set.
struct Call {
    int M, K, N, gs;
    const float *A;
    const gq4_norm *norm;  // NULL: no norm prologue
    int gate_kind;         // GateKind: the input is A gated by G
    const float *G;        // [M][K] gate vector of a gated input
    int nmat;              // 1, or 2 for gate/up
    const uint32_t *Bq[2];
    const float *scales[2];
    const float *zeros[2];
    int epi;
    float *out[4];
    int seg_start[4];
    int seg_len[4];
};

inline int prologue_of(const Call &c)
{
    return c.norm ? kProNorm
         : c.gate_kind == kGateSigmoid ? kProSigmoid
         : c.gate_kind == kGateSwiglu ? kProSwiglu
         : kProNone;
}

// CUDA-core fp32 path (any M <= GQ4_MAX_LANES).
cudaError_t launch_fp32(const Call &call, cudaStream_t stream);

// Persistent bulk-copy streaming path for one lane (M = 1).
bool stream_path_supported(const Call &call);
cudaError_t launch_stream(const Call &call, cudaStream_t stream);

// 2 <= M <= 4 lanes: persistent bulk-copy kernel, exact fp16 products on the
// warp-level MMA (K a multiple of 128 within the shared-memory plan).
bool lanes_path_supported(const Call &call);
cudaError_t launch_lanes(const Call &call, cudaStream_t stream);
cudaError_t read_lanes_device_error(unsigned int *bits, bool clear);

// bf16 tensor-core path for 16 <= M <= 32 lanes (sm_103).
bool tc_path_supported(const Call &call);
cudaError_t launch_tc(const Call &call, cudaStream_t stream);
// The same kernel for a chunk of 1..32 rows of a GEMM (fewer than 16 padded).
bool tc_rows_supported(const Call &call);

// One persistent launch for a sequence of one-lane calls (gq4_run_sequence):
// whether the calls fit its ring, and the launch (up to 128 calls per
// launch).  The workspace holds the grid barrier's counter and generation.
constexpr size_t kSeqWorkspaceBytes = 128;
constexpr int kSeqMaxCalls = 128;  // calls per persistent launch
bool sequence_plannable(const Call *calls, int n);
cudaError_t launch_sequence(const Call *calls, int n, void *workspace, cudaStream_t stream);
cudaError_t read_seq_device_error(unsigned int *bits, bool clear);
size_t seq_static_scratch_bytes();
cudaError_t seq_static_scratch(void **ptr);

// The sticky device-side error words (read, optionally clear): the one-lane
// streaming path's and the tensor-core path's.
cudaError_t read_device_error(unsigned int *bits, bool clear);
cudaError_t read_tc_device_error(unsigned int *bits, bool clear);

// The int4 GEMM for more than 32 rows (bf16 copy of A in the workspace).
size_t gemm_workspace_bytes(int M, int K);
bool gemm_path_supported(int K, int N, int gs, const float *scales, const float *zeros);
cudaError_t launch_gemm(int M, int K, int N, int gs, const float *A, const uint32_t *Bq, const float *scales,
                        const float *zeros, float *C, void *workspace, cudaStream_t stream);
cudaError_t read_gemm_device_error(unsigned int *bits, bool clear);

// Producing the format: the group-wise quantizer and the MLX converter.
cudaError_t launch_quantize(int K, int N, int gs, const float *W, uint32_t *Bq, float *scales,
                            float *zeros, cudaStream_t stream);
cudaError_t launch_from_mlx(int K, int N, int gs, const uint32_t *packed, const float *mlx_scales,
                            const float *mlx_biases, uint32_t *Bq, float *scales, float *zeros,
                            cudaStream_t stream);
cudaError_t read_quant_device_error(unsigned int *bits, bool clear);

// Int4 embedding gather.
cudaError_t launch_embedding(int T, int K, int V, int gs, const int32_t *ids, const uint32_t *Bq,
                             const float *scales, const float *zeros, float *out,
                             cudaStream_t stream);
cudaError_t read_embed_device_error(unsigned int *bits, bool clear);

// Test kernels.
cudaError_t launch_unpack(int K, int N, const uint32_t *Bq, uint8_t *q, cudaStream_t stream);
cudaError_t launch_dequant(int K, int N, int gs, const uint32_t *Bq, const float *scales,
                           const float *zeros, float *W, cudaStream_t stream);

}  // namespace gq4

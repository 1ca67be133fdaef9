// gq4_onelane.cuh -- consumer-side pieces shared by the one-lane (M = 1)
// kernels: the activation prologue and the chunk-group dot product.
//
// Activations sit in shared memory once per CTA, arranged for word_dot (see
// gq4_device.cuh): per packed word, two float4 (a0, a4, a1/16, a5/16) and
// (a2, a6, a3/16, a7/16), chunk groups XOR-swizzled by act_index so that the
// 32 lanes of a warp, reading 32 consecutive chunk groups, hit distinct
// banks.  Each chunk group also keeps the sum of its unscaled activations,
// which carries the fractional part of the zero points.  Activations are
// 16-byte aligned f32 vectors, read as float4.
//
// Operation (gerbil moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 main loop and
// WGSL_NORM_MATVEC_INT4 prologue; the GatedMatVecInt4 and SwiGLUGatedMatVecInt4
// fusion docs for the gated inputs): C[n] = sum_k a[k] * (q(n,k) - z) * s with,
// for the norm form, a = RMSNorm(A + A_b) * W_norm.
#pragma once

#include <cstdint>

#include "gq4_device.cuh"
#include "gq4_internal.h"

namespace gq4 {

// Activation loads: through the read-only path for a single call, through
// L2 only (never a possibly stale L1 line) inside a sequence of calls.
struct LoadReadOnly {
    __device__ __forceinline__ static float4 ld(const float4 *p) { return __ldg(p); }
};
struct LoadL2 {
    __device__ __forceinline__ static float4 ld(const float4 *p) { return __ldcg(p); }
};

__device__ __forceinline__ void onelane_bar(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Shared-memory slots of word u's two activation float4.
template <int R>
__device__ __forceinline__ int act_slot(int u, int half)
{
    return act_index<R>(u >> 2, 2 * (u & 3) + half);
}

// Pairs the float4 x of an even lane with its odd neighbour's (one packed
// word: a0..a3 and a4..a7) for word_dot, stores it, and stores the sum of
// each chunk group (8R consecutive float4 = 8R consecutive lanes).  All
// lanes of the warp take part; v is this lane's float4 index (v >= K4: out
// of range, x zero, nothing stored).
template <int R>
__device__ __forceinline__ void pair_and_store(float4 x, int v, int K4, int lane, float4 *s_act,
                                               float *s_asum)
{
    constexpr int kGL = 8 * R;
    const bool odd = (lane & 1) != 0;
    // the even lane keeps (a0, a4, a1, a5), the odd one (a2, a6, a3, a7)
    const float r1 = __shfl_xor_sync(0xffffffffu, odd ? x.x : x.z, 1);
    const float r2 = __shfl_xor_sync(0xffffffffu, odd ? x.y : x.w, 1);
    const float4 pr = odd ? make_float4(r1, x.z, r2 * 0.0625f, x.w * 0.0625f)
                          : make_float4(x.x, r1, x.y * 0.0625f, r2 * 0.0625f);
    float a = (x.x + x.y) + (x.z + x.w);
#pragma unroll
    for (int off = 1; off < kGL; off <<= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if (v < K4) {
        s_act[act_slot<R>(v >> 1, v & 1)] = pr;
        if ((lane & (kGL - 1)) == 0) s_asum[v / kGL] = a;
    }
}

// One element of a gated input: x * sigmoid(g) (kProSigmoid) or silu(g) * x
// (kProSwiglu), with sigmoid(g) = 1 / (1 + e^-g) and silu(g) = g sigmoid(g).
// The fast exponential and divide intrinsics: a few ulp, far inside the
// matvec's tolerance; a saturated gate (e^-g = inf) gives exactly 0.
template <int PRO>
__device__ __forceinline__ float gate_input(float x, float g)
{
    if constexpr (PRO == kProSigmoid)
        return __fdividef(x, 1.0f + __expf(-g));
    else
        return __fdividef(g, 1.0f + __expf(-g)) * x;
}

// Stages one call's activations (K a multiple of 32; K/32 even when R = 2)
// and the chunk groups' activation sums.  NT consumer threads (ctid < NT)
// take part; named barrier `bar_id` synchronises them.  PRO (Prologue):
//   kProNone     a = A;
//   kProNorm     x = A + A_b (A_b may be null), a = x / sqrt(mean(x^2) + eps)
//                * W_norm; when `side_outputs`, x is written to residual_out
//                and a to norm_out (either may be null);
//   kProSigmoid  a = A * sigmoid(A_b)   (A_b is the gate vector);
//   kProSwiglu   a = silu(A_b) * A      (A_b is the gate vector).
// s_norm holds NT/32 floats.
//
// Consecutive lanes own consecutive float4 of the vector (coalesced loads),
// up to NV per thread per batch, all issued before any use: for K <= 4*NV*NT
// the whole prologue pays one round trip to L2 (the norm gain included).
// Longer vectors take several batches; with the norm, x then waits in shared
// memory for the inverse RMS.
template <int R, int PRO, int NT, int NV, class Ld>
__device__ __forceinline__ void stage_activations(int K, const float *A, const float *A_b,
                                                  const float *W_norm, float eps, float *residual_out,
                                                  float *norm_out, bool side_outputs, float4 *s_act,
                                                  float *s_asum, float *s_norm, int ctid, int bar_id)
{
    constexpr int kWarps = NT / 32;
    constexpr int kBatch = NV * NT;
    const int K4 = K >> 2;
    const int lane = ctid & 31;
    const float4 *A4 = reinterpret_cast<const float4 *>(A);
    const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if constexpr (PRO == kProNorm) {
        const float4 *B4 = reinterpret_cast<const float4 *>(A_b);
        const float4 *W4 = reinterpret_cast<const float4 *>(W_norm);
        const bool one_batch = K4 <= kBatch;
        float4 *res4 = side_outputs ? reinterpret_cast<float4 *>(residual_out) : nullptr;
        float4 x[NV], g[NV];
        float part = 0.0f;
        for (int b0 = 0; b0 < K4; b0 += kBatch) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = b0 + ctid + i * NT;
                x[i] = v < K4 ? Ld::ld(A4 + v) : z4;
                const float4 b = (v < K4 && B4) ? Ld::ld(B4 + v) : z4;
                if (b0 == 0) g[i] = v < K4 ? Ld::ld(W4 + v) : z4;
                x[i].x += b.x; x[i].y += b.y; x[i].z += b.z; x[i].w += b.w;
            }
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = b0 + ctid + i * NT;
                if (v - lane >= K4) break;  // warp-uniform: the rest of the batch is past the end
                if (v < K4) {
                    if (res4) res4[v] = x[i];
                    // several batches: x waits in shared memory (natural order)
                    if (!one_batch) s_act[act_slot<R>(v >> 1, v & 1)] = x[i];
                }
                part = fmaf(x[i].x, x[i].x, part);
                part = fmaf(x[i].y, x[i].y, part);
                part = fmaf(x[i].z, x[i].z, part);
                part = fmaf(x[i].w, x[i].w, part);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) s_norm[ctid >> 5] = part;
        onelane_bar(bar_id, NT);
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += s_norm[w];
        const float inv = 1.0f / sqrtf(sum / (float)K + eps);
        float4 *nrm4 = side_outputs ? reinterpret_cast<float4 *>(norm_out) : nullptr;
        for (int b0 = 0; b0 < K4; b0 += kBatch) {
            if (!one_batch) {
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int v = b0 + ctid + i * NT;
                    x[i] = v < K4 ? s_act[act_slot<R>(v >> 1, v & 1)] : z4;
                    if (b0 > 0) g[i] = v < K4 ? Ld::ld(W4 + v) : z4;
                }
                // every lane has read its own slots before any pair is written
                __syncwarp();
            }
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = b0 + ctid + i * NT;
                if (v - lane >= K4) break;  // warp-uniform: the rest of the batch is past the end
                x[i].x = (x[i].x * inv) * g[i].x;
                x[i].y = (x[i].y * inv) * g[i].y;
                x[i].z = (x[i].z * inv) * g[i].z;
                x[i].w = (x[i].w * inv) * g[i].w;
                if (nrm4 && v < K4) nrm4[v] = x[i];
                pair_and_store<R>(x[i], v, K4, lane, s_act, s_asum);
            }
        }
    } else {
        const float4 *G4 = reinterpret_cast<const float4 *>(A_b);
        for (int b0 = 0; b0 < K4; b0 += kBatch) {
            float4 x[NV];
            float4 g[PRO == kProNone ? 1 : NV];
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = b0 + ctid + i * NT;
                x[i] = v < K4 ? Ld::ld(A4 + v) : z4;
                if constexpr (PRO != kProNone) g[i] = v < K4 ? Ld::ld(G4 + v) : z4;
            }
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int v = b0 + ctid + i * NT;
                if (v - lane >= K4) break;  // warp-uniform: the rest of the batch is past the end
                if constexpr (PRO != kProNone) {
                    // the gated input: x * sigmoid(g), or silu(g) * x
                    x[i].x = gate_input<PRO>(x[i].x, g[i].x);
                    x[i].y = gate_input<PRO>(x[i].y, g[i].y);
                    x[i].z = gate_input<PRO>(x[i].z, g[i].z);
                    x[i].w = gate_input<PRO>(x[i].w, g[i].w);
                }
                pair_and_store<R>(x[i], v, K4, lane, s_act, s_asum);
            }
        }
    }
    onelane_bar(bar_id, NT);
}

// One chunk group (R consecutive 32-code chunks, one scale group) of SPW
// weight streams: acc[q] += sc[q] * (sum_k a_k (q_k - zi) + dz * sum_k a_k).
// Two accumulators per stream (words 0-1 and 2-3 of each chunk).
template <int SPW, int R>
__device__ __forceinline__ void chunk_group_dot(const float4 *s_act, int jg, float asum,
                                                const uint4 (&wq)[SPW][R], const float (&sc)[SPW],
                                                const HalfZero (&hz)[SPW], uint32_t magic,
                                                float (&acc)[SPW])
{
    f32x2 in0[SPW], in1[SPW];
#pragma unroll
    for (int q = 0; q < SPW; ++q) {
        in0[q] = pack2(0.0f, 0.0f);
        in1[q] = pack2(0.0f, 0.0f);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        // the chunk's 32 activations, loaded before any use
        ulonglong2 av[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            av[j] = reinterpret_cast<const ulonglong2 *>(s_act)[act_index<R>(jg * R + r, j)];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
            for (int q = 0; q < SPW; ++q) {
                const uint32_t word = wd == 0 ? wq[q][r].x : wd == 1 ? wq[q][r].y
                                    : wd == 2 ? wq[q][r].z : wq[q][r].w;
                if (wd < 2)
                    in0[q] = word_dot(word, av[2 * wd], av[2 * wd + 1], hz[q], magic, in0[q]);
                else
                    in1[q] = word_dot(word, av[2 * wd], av[2 * wd + 1], hz[q], magic, in1[q]);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < SPW; ++q) {
        const float2 v = unpack2(add2(in0[q], in1[q]));
        acc[q] = fmaf(sc[q], fmaf(hz[q].dz, asum, v.x + v.y), acc[q]);
    }
}

}  // namespace gq4

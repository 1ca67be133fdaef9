// gq4_onelane.cuh -- consumer-side pieces shared by the one-lane (M = 1)
// kernels: the activation prologue and the chunk-group dot product.
//
// Activations sit in shared memory once per CTA, arranged for word_dot (see
// gq4_device.cuh): per packed word, two float4 (a0, a4, a1/16, a5/16) and
// (a2, a6, a3/16, a7/16), chunk groups XOR-swizzled by act_index so that the
// 32 lanes of a warp, reading 32 consecutive chunk groups, hit distinct
// banks.  Each chunk group also keeps the sum of its unscaled activations,
// which carries the fractional part of the zero points.
//
// Operation (gerbil moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 main loop and
// WGSL_NORM_MATVEC_INT4 prologue): C[n] = sum_k a[k] * (q(n,k) - z) * s with,
// for the norm form, a = RMSNorm(A + A_b) * W_norm.
#pragma once

#include <cstdint>

#include "gq4_device.cuh"

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

// Stages one call's activations (K a multiple of 32) and the chunk groups'
// activation sums.  NT consumer threads (ctid < NT) take part; named barrier
// `bar_id` synchronises them.  NORM: x = A + A_b (A_b may be null), then
// a = x / sqrt(mean(x^2) + eps) * W_norm; when `side_outputs`, x is written to
// residual_out and a to norm_out (either may be null).  Loads are issued in
// batches of several words per thread before any use, so their latency is
// paid once per batch.  s_norm holds NT/32 floats.
template <int R, bool NORM, int NT, class Ld>
__device__ __forceinline__ void stage_activations(int K, int KP, const float *A, const float *A_b,
                                                  const float *W_norm, float eps, float *residual_out,
                                                  float *norm_out, bool side_outputs, float4 *s_act,
                                                  float *s_asum, float *s_norm, int ctid, int bar_id)
{
    constexpr int kB = NORM ? 3 : 6;  // words per thread per batch
    constexpr int kWarps = NT / 32;
    const int Kw = K >> 3;  // packed words per column
    const float4 *A4 = reinterpret_cast<const float4 *>(A);
    const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if constexpr (NORM) {
        const float4 *B4 = reinterpret_cast<const float4 *>(A_b);
        float part = 0.0f;
        float4 *res4 = side_outputs ? reinterpret_cast<float4 *>(residual_out) : nullptr;
        for (int u0 = ctid; u0 < Kw; u0 += kB * NT) {
            float4 x[kB][2], b[kB][2];
#pragma unroll
            for (int i = 0; i < kB; ++i) {
                const int u = u0 + i * NT;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    x[i][h] = u < Kw ? Ld::ld(A4 + 2 * u + h) : z4;
                    b[i][h] = (u < Kw && B4) ? Ld::ld(B4 + 2 * u + h) : z4;
                }
            }
#pragma unroll
            for (int i = 0; i < kB; ++i) {
                const int u = u0 + i * NT;
                if (u >= Kw) continue;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float4 &v = x[i][h];
                    v.x += b[i][h].x; v.y += b[i][h].y; v.z += b[i][h].z; v.w += b[i][h].w;
                    if (res4) res4[2 * u + h] = v;
                    part = fmaf(v.x, v.x, part);
                    part = fmaf(v.y, v.y, part);
                    part = fmaf(v.z, v.z, part);
                    part = fmaf(v.w, v.w, part);
                    s_act[act_slot<R>(u, h)] = v;  // natural order, unscaled for now
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if ((ctid & 31) == 0) s_norm[ctid >> 5] = part;
        onelane_bar(bar_id, NT);
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += s_norm[w];
        const float inv = 1.0f / sqrtf(sum / (float)K + eps);
        float4 *nrm4 = side_outputs ? reinterpret_cast<float4 *>(norm_out) : nullptr;
        const float4 *W4 = reinterpret_cast<const float4 *>(W_norm);
        for (int u0 = ctid; u0 < Kw; u0 += kB * NT) {
            float4 g[kB][2];
#pragma unroll
            for (int i = 0; i < kB; ++i) {
                const int u = u0 + i * NT;
#pragma unroll
                for (int h = 0; h < 2; ++h) g[i][h] = u < Kw ? Ld::ld(W4 + 2 * u + h) : z4;
            }
#pragma unroll
            for (int i = 0; i < kB; ++i) {
                const int u = u0 + i * NT;
                if (u >= Kw) continue;
                float4 a[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 v = s_act[act_slot<R>(u, h)];
                    a[h].x = (v.x * inv) * g[i][h].x;
                    a[h].y = (v.y * inv) * g[i][h].y;
                    a[h].z = (v.z * inv) * g[i][h].z;
                    a[h].w = (v.w * inv) * g[i][h].w;
                    if (nrm4) nrm4[2 * u + h] = a[h];
                }
                float4 lo, hi;
                pair_activations(a[0], a[1], lo, hi);
                s_act[act_slot<R>(u, 0)] = lo;
                s_act[act_slot<R>(u, 1)] = hi;
            }
        }
    } else {
        for (int u0 = ctid; u0 < Kw; u0 += kB * NT) {
            float4 x[kB][2];
#pragma unroll
            for (int i = 0; i < kB; ++i) {
                const int u = u0 + i * NT;
#pragma unroll
                for (int h = 0; h < 2; ++h) x[i][h] = u < Kw ? Ld::ld(A4 + 2 * u + h) : z4;
            }
#pragma unroll
            for (int i = 0; i < kB; ++i) {
                const int u = u0 + i * NT;
                if (u >= Kw) continue;
                float4 lo, hi;
                pair_activations(x[i][0], x[i][1], lo, hi);
                s_act[act_slot<R>(u, 0)] = lo;
                s_act[act_slot<R>(u, 1)] = hi;
            }
        }
    }
    onelane_bar(bar_id, NT);
    // activation sum of each chunk group (unscaled, fixed order)
    for (int jg = ctid; jg < KP; jg += NT) {
        float a = 0.0f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int j = 0; j < 8; ++j) a += paired_sum(s_act[act_index<R>(jg * R + r, j)]);
        }
        s_asum[jg] = a;
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

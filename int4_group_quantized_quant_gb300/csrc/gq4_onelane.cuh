// gq4_onelane.cuh -- consumer-side pieces shared by the one-lane (M = 1)
// kernels: the activation prologue and the chunk-group dot product, in the
// integer form of gq4_device.cuh (word_dot_i8).
//
// Activations sit in shared memory once per CTA as 24-bit fixed-point
// integers with a power-of-two scale per chunk group (R consecutive 32-code
// chunks of one scale group), split into three byte pieces and arranged per
// packed word for dp4a; chunks are XOR-swizzled by act_index so that the 32
// lanes of a warp, reading 32 consecutive chunk groups, hit distinct banks.
// Each chunk group also keeps its piece sums (the integer part of the zero
// points comes off through them) and the f32 sum of its activations (which
// carries the fractional part).  Activations are 16-byte aligned f32
// vectors, read as float4.
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

}  // namespace gq4

namespace gq4 {

// ===========================================================================
// Integer form of the one-lane dot product (word_dot_i8, gq4_device.cuh).
//
// Shared-memory layout of the staged activations: chunk t (32 codes, four
// packed words) takes 128 bytes, eight uint4 slots, slot j stored at
// act_index<R>(t, j) (XOR-swizzled per chunk group, conflict-free for 32
// lanes reading 32 consecutive chunk groups):
//   slots 0..5  the piece words E2, O2, E1, O1, E0, O0 of the chunk's four
//               packed words (uint4 component u = word u): byte j of E_p is
//               piece p of activation 8u + 2j, of O_p of activation 8u + 2j + 1;
//   slot 6      (first chunk of each chunk group) the group's piece sums
//               {sum B2, sum B1, sum B0} and the f32 sum of its activations;
//   slot 7      (first chunk of each chunk group) 2^(E-26), E its exponent.
// ===========================================================================

// Quantizes NQ float4 per thread (float4 index v0 + i * stride for x[i],
// activations 4v .. 4v+3) into the layout above.  All lanes of the warp take
// part (v >= K4: out of range, x zero, nothing stored); 8R consecutive
// lanes hold one chunk group.  The NQ items' shuffle chains are independent
// and interleaved.
template <int R, int NQ>
__device__ __forceinline__ void quantize_and_store_i8(const float4 (&x)[NQ], int v0, int stride, int K4,
                                                      int lane, uint4 *s_act)
{
    constexpr int kGL = 8 * R;
    float mx[NQ], sm[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        mx[i] = fmaxf(fmaxf(fabsf(x[i].x), fabsf(x[i].y)), fmaxf(fabsf(x[i].z), fabsf(x[i].w)));
        sm[i] = (x[i].x + x[i].y) + (x[i].z + x[i].w);
    }
#pragma unroll
    for (int off = 1; off < kGL; off <<= 1) {
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], off));
            sm[i] += __shfl_xor_sync(0xffffffffu, sm[i], off);
        }
    }
    int X[NQ][4];
    int sB2[NQ], sB10[NQ];
    float fac16[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        // the group's exponent: max |a| < 2^E (zero or subnormal maxima
        // clamp).  A non-finite activation makes the group's value NaN: an
        // infinite maximum gives it a NaN scale, and a NaN (which the max
        // skips) makes sm NaN, which reaches the value through dz * asum.
        int E = (int)(__float_as_uint(mx[i]) >> 23) - 126;
        E = min(max(E, -100), 127);
        const float sc = __uint_as_float((uint32_t)(149 - E) << 23);  // 2^(22 - E)
        fac16[i] = __float_as_uint(mx[i]) >= 0x7f800000u ? __uint_as_float(0x7fffffffu)
                                                         : __uint_as_float((uint32_t)(E + 101) << 23);  // 2^(E - 26)
        X[i][0] = __float_as_int(__fmaf_rn(x[i].x, sc, kI8MagicF)) - kI8Magic;
        X[i][1] = __float_as_int(__fmaf_rn(x[i].y, sc, kI8MagicF)) - kI8Magic;
        X[i][2] = __float_as_int(__fmaf_rn(x[i].z, sc, kI8MagicF)) - kI8Magic;
        X[i][3] = __float_as_int(__fmaf_rn(x[i].w, sc, kI8MagicF)) - kI8Magic;
        // B2 sums, and the B1 and B0 sums packed in one word (each below 2^16)
        sB2[i] = 0;
        sB10[i] = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sB2[i] += X[i][j] >> 16;
            sB10[i] += (int)(((uint32_t)X[i][j] & 0xFF00u) << 8) + (X[i][j] & 0xFF);
        }
    }
#pragma unroll
    for (int off = 1; off < kGL; off <<= 1) {
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            sB2[i] += __shfl_xor_sync(0xffffffffu, sB2[i], off);
            sB10[i] += __shfl_xor_sync(0xffffffffu, sB10[i], off);
        }
    }
    uint32_t *s32 = reinterpret_cast<uint32_t *>(s_act);
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        const int v = v0 + i * stride;
        const bool odd = (v & 1) != 0;
        // piece p's bytes of (X0, X2 | X1, X3): the even and the odd codes' halves
        uint32_t word[3];
#pragma unroll
        for (int p = 0; p < 3; ++p) {
            const uint32_t b = (uint32_t)(2 - p);  // byte 2 = B2, 1 = B1, 0 = B0
            const uint32_t sel = b | ((b + 4u) << 4);
            const uint32_t ev = __byte_perm((uint32_t)X[i][0], (uint32_t)X[i][2], sel);
            const uint32_t od = __byte_perm((uint32_t)X[i][1], (uint32_t)X[i][3], sel);
            const uint32_t pk = __byte_perm(ev, od, 0x5410);
            const uint32_t pp = __shfl_xor_sync(0xffffffffu, pk, 1);
            // the even lane keeps the E word, the odd lane the O word
            word[p] = odd ? __byte_perm(pp, pk, 0x7632) : __byte_perm(pk, pp, 0x5410);
        }
        if (v < K4) {
            const int t = v >> 3;        // chunk
            const int u = (v >> 1) & 3;  // word within the chunk
#pragma unroll
            for (int p = 0; p < 3; ++p) s32[act_index<R>(t, 2 * p + (odd ? 1 : 0)) * 4 + u] = word[p];
            if ((lane & (kGL - 1)) == 0) {
                const int t0 = (v / kGL) * R;
                s_act[act_index<R>(t0, 6)] =
                    make_uint4((uint32_t)sB2[i], (uint32_t)sB10[i] >> 16, (uint32_t)sB10[i] & 0xFFFFu,
                               __float_as_uint(sm[i]));
                s_act[act_index<R>(t0, 7)] = make_uint4(__float_as_uint(fac16[i]), 0u, 0u, 0u);
            }
        }
    }
}

// Stages one call's activations in the integer layout (K a multiple of 32;
// K/32 even when R = 2).  NT consumer threads (ctid < NT) take part; named
// barrier `bar_id` synchronises them.  PRO (Prologue):
//   kProNone     a = A;
//   kProNorm     x = A + A_b (A_b may be null), a = x * W_norm: the inverse
//                RMS 1 / sqrt(mean(x^2) + eps) is returned, a scalar that the
//                caller applies to each finished dot product; when
//                `side_outputs`, x is written to residual_out (if not null);
//   kProSigmoid  a = A * sigmoid(A_b)   (A_b is the gate vector);
//   kProSwiglu   a = silu(A_b) * A      (A_b is the gate vector).
// Returns 1 for the other prologues.  s_norm holds NT/32 floats.
// Consecutive lanes own consecutive float4 (coalesced loads), NV per thread
// per batch, all issued before any use.
template <int R, int PRO, int NT, int NV, class Ld>
__device__ __forceinline__ float stage_activations_i8(int K, const float *A, const float *A_b,
                                                      const float *W_norm, float eps, float *residual_out,
                                                      bool side_outputs, uint4 *s_act, float *s_norm,
                                                      int ctid, int bar_id)
{
    constexpr int kWarps = NT / 32;
    constexpr int kBatch = NV * NT;
    const int K4 = K >> 2;
    const int lane = ctid & 31;
    const float4 *A4 = reinterpret_cast<const float4 *>(A);
    const float4 *B4 = reinterpret_cast<const float4 *>(A_b);
    const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float4 *res4 = (PRO == kProNorm && side_outputs) ? reinterpret_cast<float4 *>(residual_out) : nullptr;
    float part = 0.0f;
    for (int b0 = 0; b0 < K4; b0 += kBatch) {
        float4 x[NV];
        float4 g[PRO == kProNone ? 1 : NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int v = b0 + ctid + i * NT;
            x[i] = v < K4 ? Ld::ld(A4 + v) : z4;
            if constexpr (PRO == kProNorm) {
                const float4 b = (v < K4 && B4) ? Ld::ld(B4 + v) : z4;
                g[i] = v < K4 ? Ld::ld(reinterpret_cast<const float4 *>(W_norm) + v) : z4;
                x[i].x += b.x; x[i].y += b.y; x[i].z += b.z; x[i].w += b.w;
            } else if constexpr (PRO != kProNone) {
                g[i] = v < K4 ? Ld::ld(B4 + v) : z4;
            }
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int v = b0 + ctid + i * NT;
            if constexpr (PRO == kProNorm) {
                if (res4 && v < K4) res4[v] = x[i];
                part = fmaf(x[i].x, x[i].x, part);
                part = fmaf(x[i].y, x[i].y, part);
                part = fmaf(x[i].z, x[i].z, part);
                part = fmaf(x[i].w, x[i].w, part);
                x[i].x *= g[i].x; x[i].y *= g[i].y; x[i].z *= g[i].z; x[i].w *= g[i].w;
            } else if constexpr (PRO != kProNone) {
                x[i].x = gate_input<PRO>(x[i].x, g[i].x);
                x[i].y = gate_input<PRO>(x[i].y, g[i].y);
                x[i].z = gate_input<PRO>(x[i].z, g[i].z);
                x[i].w = gate_input<PRO>(x[i].w, g[i].w);
            }
        }
        // quantize in groups of four float4, the warp-uniform rest past the end skipped
        constexpr int kQ = 4;
        static_assert(NV % kQ == 0, "prologue batch must be a multiple of 4 float4");
#pragma unroll
        for (int i0 = 0; i0 < NV; i0 += kQ) {
            if (b0 + (ctid - lane) + i0 * NT >= K4) break;  // warp-uniform
            float4 xq[kQ];
#pragma unroll
            for (int i = 0; i < kQ; ++i) xq[i] = x[i0 + i];
            quantize_and_store_i8<R, kQ>(xq, b0 + ctid + i0 * NT, NT, K4, lane, s_act);
        }
    }
    if constexpr (PRO == kProNorm) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) s_norm[ctid >> 5] = part;
    }
    onelane_bar(bar_id, NT);
    if constexpr (PRO == kProNorm) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += s_norm[w];
        return 1.0f / sqrtf(sum / (float)K + eps);
    } else {
        return 1.0f;
    }
}

// norm_out = (x * inv) * W_norm with x = A + A_b, written by NT threads
// (after the dot products, so that it does not delay them).
template <int NT, class Ld>
__device__ __forceinline__ void write_norm_out(int K, const float *A, const float *A_b, const float *W_norm,
                                               float inv, float *norm_out, int ctid)
{
    const int K4 = K >> 2;
    const float4 *A4 = reinterpret_cast<const float4 *>(A);
    const float4 *B4 = reinterpret_cast<const float4 *>(A_b);
    const float4 *W4 = reinterpret_cast<const float4 *>(W_norm);
    float4 *n4 = reinterpret_cast<float4 *>(norm_out);
    for (int v = ctid; v < K4; v += NT) {
        float4 x = Ld::ld(A4 + v);
        if (B4) {
            const float4 b = Ld::ld(B4 + v);
            x.x += b.x; x.y += b.y; x.z += b.z; x.w += b.w;
        }
        const float4 g = Ld::ld(W4 + v);
        n4[v] = make_float4((x.x * inv) * g.x, (x.y * inv) * g.y, (x.z * inv) * g.z, (x.w * inv) * g.w);
    }
}

// Chunk order within a chunk group for lane `lane`: with R = 2, lanes 4..7
// of every 8 take the group's two chunks in the other order, so that the
// eight lanes of one 128-bit shared-memory phase hit eight distinct bank
// groups (the integer sums do not depend on the order).
template <int R>
__device__ __forceinline__ int chunk_swap(int lane)
{
    return R == 2 ? ((lane >> 2) & 1) : 0;
}

// One chunk group (R chunks, one scale group) of SPW weight streams:
// acc[q] += sc[q] * sum_k a_k (q_k - z[q]).  wq[q][r] holds chunk
// jg*R + (r ^ chunk_swap) of stream q.
template <int SPW, int R>
__device__ __forceinline__ void chunk_group_dot_i8(const uint4 *s_act, int jg, int swap,
                                                   const uint4 (&wq)[SPW][R], const float (&sc)[SPW],
                                                   const float (&zz)[SPW], uint32_t mask, float (&acc)[SPW])
{
    const int t0 = jg * R;
    const uint4 meta = s_act[act_index<R>(t0, 6)];
    const float fac16 = __uint_as_float(s_act[act_index<R>(t0, 7)].x);
    const int sB[3] = {(int)meta.x, (int)meta.y, (int)meta.z};
    const float asum = __uint_as_float(meta.w);
    I8Acc a[SPW];
    IntZero iz[SPW];
#pragma unroll
    for (int q = 0; q < SPW; ++q) {
        iz[q] = int_zero(zz[q]);
        int_group_init(a[q], iz[q].zi, sB);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int t = t0 + (r ^ swap);
        uint4 av[6];
#pragma unroll
        for (int j = 0; j < 6; ++j) av[j] = s_act[act_index<R>(t, j)];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
            for (int q = 0; q < SPW; ++q) {
                const uint32_t word = wd == 0 ? wq[q][r].x : wd == 1 ? wq[q][r].y
                                    : wd == 2 ? wq[q][r].z : wq[q][r].w;
#define GQ4_C(v) (wd == 0 ? (v).x : wd == 1 ? (v).y : wd == 2 ? (v).z : (v).w)
                word_dot_i8(word, mask, GQ4_C(av[0]), GQ4_C(av[1]), GQ4_C(av[2]), GQ4_C(av[3]),
                            GQ4_C(av[4]), GQ4_C(av[5]), a[q]);
#undef GQ4_C
            }
        }
    }
#pragma unroll
    for (int q = 0; q < SPW; ++q) acc[q] = fmaf(sc[q], int_group_value(a[q], fac16, iz[q].dz, asum), acc[q]);
}

}  // namespace gq4

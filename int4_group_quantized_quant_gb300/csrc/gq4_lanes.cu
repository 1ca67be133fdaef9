// gq4_lanes.cu -- persistent, bulk-copy fed kernels for 2 to 4 decode lanes
// (2 <= M <= 4): plain, quad routing, RMSNorm prologue, gated inputs,
// SiLU-gated gate/up and dual, dot products on the tensor cores' legacy
// warp-level MMA, exactly in the products.
//
// Operation (gerbil moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 and
// WGSL_NORM_MATVEC_INT4; the DualMatVecInt4, GatedMatVecInt4 and
// SwiGLUGatedMatVecInt4 fusion docs): C[m][n] = sum_k a[m][k] * (q(n,k) - z) * s,
// a built by the call's prologue; two matrices for gate/up or dual.
//
// Arithmetic.  Per lane the work equals the one-lane path's, so a CUDA-core
// dot product costs M times as much; here the weight codes are decoded once
// for all lanes and the lanes ride in the N columns of one MMA:
//   * A bit mask moves two codes of a packed word into the two fp16 halves of
//     a register: bits 0-3 and 16-19 give the fp16 bit patterns q, read as the
//     subnormal values q * 2^-24 exactly; bits 4-7 and 20-23 give 16 q * 2^-24.
//     A shift by 8 brings the other four codes of the word to the same places.
//     The integer part zi of the zero point comes off in fp16 (zi * 2^-24 and
//     16 zi * 2^-24 are subnormals too, and the differences are exact), so
//     codes equal to an integer zero contribute exactly nothing.
//   * Activations are staged per lane and 128-code block, scaled by a power of
//     two so the block's largest magnitude lies in [2^13, 2^14), as an fp16
//     high part and an fp16 low part (x' = hi + lo to about 22 bits); the
//     odd code positions take x' / 16, matching the 16 q of their codes.
//   * mma.sync m16n8k16 (fp16 inputs, f32 accumulation): 16 weight columns
//     (rows of the MMA) times 8 columns of B = {hi, lo} of 4 lanes.  Products
//     of the fp16 operands are exact; the sums are f32.
//   * Per block, column and lane: y += s * (2^(24-e) D - (z - zi) X), with D
//     the MMA sum of (q - zi) x' over the block, e the block's scale exponent
//     and X the f32 sum of the block's activations (the fractional part of the
//     zero point comes off through X).
//
// Decomposition:
//   * Persistent grid, one CTA per SM, a contiguous range of whole columns per
//     CTA (balanced in units whose scale/zero rows start 16-byte aligned).
//   * One producer warp streams the CTA's scale/zero rows once, then the codes
//     through a ring of stages.  A stage is one MMA tile: 16 columns (8 gate
//     and 8 up columns for gate/up, 8 and 8 of the two matrices for dual),
//     fetched as two bulk copies of 8 whole columns into two regions whose
//     bases differ by 64 bytes mod 128, so that MMA rows g and g + 1 (lanes
//     4g.. and 4g+4..) read disjoint bank halves.
//   * The 8 consumer warps split each stage's K into 8 slices of whole
//     128-code blocks.  Per stage a warp first copies the scale and zero of
//     its groups for the tile's 16 columns into a private scratch area laid
//     out for conflict-free reads, then runs its blocks; its partial sums go
//     to a per-ring-entry buffer and the last warp to finish the stage (a
//     shared counter) adds the 8 partials in warp order and writes the
//     outputs.  A ring entry is released only after that sum, so the next
//     occupant cannot overwrite the partials early.
//   * Programmatic dependent launch as in the one-lane kernel: the producer
//     streams weights before the dependency wait, the consumers wait before
//     reading activations; a kernel signals its dependents at its last stage.
//   * Every mbarrier wait is bounded in time; on expiry the kernel records an
//     error in a device word (gq4_device_error), writes NaN and releases its
//     stages.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gq4_device.cuh"
#include "gq4_host.h"
#include "gq4_internal.h"
#include "gq4_onelane.cuh"
#include "gq4_tma.cuh"

namespace gq4 {

// Sticky device-side error word of this path (bit 5: a wait timed out).
__device__ unsigned int g_lanes_error = 0;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kCT = kConsumerWarps * 32;
constexpr int kMaxStages = 16;
constexpr int kBlock = 128;  // codes per activation block (one scale exponent, one MMA run)
constexpr uint32_t kSmemLimit = 220u * 1024u;

struct LanesParams {
    int M, K, N, gs;
    int KW;          // packed words per column (K / 8)
    int KB;          // 128-code blocks per column
    int G;           // scale groups per column
    int bpg;         // blocks per scale group (gs / 128)
    int S;           // ring depth
    int unit;        // column granularity of the balanced split
    int n_units;
    int max_groups;  // most groups any warp's K slice touches (scratch rows)
    uint32_t col_bytes;    // bytes of one column's codes (K / 2)
    uint32_t stage_bytes;
    uint32_t off_reg1;     // second region of a stage (64 mod 128)
    uint32_t off_s[2], off_z[2];  // scale/zero rows of the CTA's range (per matrix)
    uint32_t off_act, off_fx, off_part, off_scr, off_misc, off_bar;
    const float *A;
    const float *A_b;
    const float *W_norm;
    float eps;
    float *residual_out;
    float *norm_out;
    const uint4 *Bq[2];
    const float *scales[2];
    const float *zeros[2];
    float *out[4];
    int seg_start[4];
    int seg_len[4];
};

__device__ __forceinline__ void lanes_bar(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void lanes_bar_arrive(int id, int threads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void lanes_dependents_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void lanes_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void lanes_error()
{
    atomicOr(&g_lanes_error, 32u);
}

// D += A B for one m16n8k16 tile: A 16 x 16 fp16 (row-major fragments a0..a3),
// B 16 x 8 fp16 (b0, b1), D 16 x 8 f32.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^k as an f32 for -126 <= k <= 127 (exact).
__device__ __forceinline__ float pow2i(int k)
{
    return __int_as_float((k + 127) << 23);
}

// x * 2^k, exact unless the result leaves the f32 range, for |k| <= 252.
__device__ __forceinline__ float mul_pow2(float x, int k)
{
    const int k1 = k / 2;
    return (x * pow2i(k1)) * pow2i(k - k1);
}

// a - b on two fp16 halves (round to nearest, subnormals kept: the operands
// here are subnormal integers times 2^-24 and the difference is exact).
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h)
{
    return *reinterpret_cast<uint32_t *>(&h);
}

// fp16 high and low parts of two values (low halves: a, high halves: b).
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo)
{
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
    hi = h2_bits(h);
    lo = h2_bits(l);
}

// One packed word w of lane m in the prologue: its 8 activations x (zero
// for a word past K or a lane past M), the block's largest magnitude and sum
// over the 16 lanes holding the block (all 32 lanes of the warp call this
// together), the power-of-two scale, and the fp16 high/low parts stored in
// the MMA's B layout [block][pair][n = 2m + part][t][8 halves]; the block's
// {f1, f2, X} (f1 f2 = 2^(24 - k), X = sum of x) by its first lane.
template <int NP>
__device__ __forceinline__ void stage_word(const float (&x)[8], int m, int w, bool ok, int lane,
                                           unsigned char *s_act, unsigned char *s_fx)
{
    float mx = 0.0f, sm = 0.0f;
    bool bad = false;  // inf or NaN (fmaxf would drop a NaN)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        mx = fmaxf(mx, fabsf(x[j]));
        sm += x[j];
        bad |= !(fabsf(x[j]) <= 3.402823466e38f);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        sm += __shfl_xor_sync(0xffffffffu, sm, off);
        bad |= __shfl_xor_sync(0xffffffffu, (int)bad, off) != 0;
    }
    float f1, f2;
    int k;  // x' = x 2^k
    if (bad) {
        f1 = __int_as_float(0x7fffffff);  // the block's lane results become NaN
        f2 = 1.0f;
        k = 0;
    } else if (mx == 0.0f) {
        f1 = 0.0f;
        f2 = 0.0f;
        k = 0;
    } else {
        const int E = ilogbf(mx);  // mx in [2^E, 2^(E+1))
        k = 13 - E;
        const int j = 11 + E;      // 2^(24 - k)
        const int j1 = j / 2;
        f1 = pow2i(j1);
        f2 = pow2i(j - j1);
    }
    float xs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float v = bad ? 0.0f : mul_pow2(x[j], k);
        xs[j] = (j & 1) ? v * 0.0625f : v;
    }
    if (!ok) return;
    uint4 hi, lo;
    split_pair(xs[0], xs[4], hi.x, lo.x);
    split_pair(xs[1], xs[5], hi.y, lo.y);
    split_pair(xs[2], xs[6], hi.z, lo.z);
    split_pair(xs[3], xs[7], hi.w, lo.w);
    const int b = w >> 4, wi = w & 15;
    const int t = wi >> 2, pr = wi & 3;
    uint4 *dst = reinterpret_cast<uint4 *>(s_act + ((size_t)(b * 4 + pr) * (2 * NP) + 2 * m) * 64 + t * 16);
    dst[0] = hi;
    dst[4] = lo;  // n = 2m + 1: 64 bytes on
    if ((lane & 15) == 0)
        *reinterpret_cast<float4 *>(s_fx + ((size_t)b * 4 + m) * 16) = make_float4(f1, f2, sm, 0.0f);
}

// NP: lanes per MMA (2 or 4; the N columns are {hi, lo} of each lane).
template <int NMAT, int PRO, int EPI, int NP>
__global__ void __launch_bounds__(kThreads, 1) lanes_matvec_kernel(const __grid_constant__ LanesParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + kMaxStages;
    uint64_t *srows = empty + kMaxStages;  // scale/zero rows landed
    uint64_t *ready = srows + 1;           // consumers' prologue done
    int *s_seq = reinterpret_cast<int *>(ready + 1);  // stage a ring entry holds
    int *s_cnt = s_seq + kMaxStages;                  // warps done with a ring entry
    float *s_inv = reinterpret_cast<float *>(smem + p.off_misc);        // [4] inverse RMS per lane
    float *s_sq = s_inv + 4;                                            // [8 warps][4] square sums
    unsigned char *s_act = smem + p.off_act;
    const float4 *s_fx = reinterpret_cast<const float4 *>(smem + p.off_fx);  // [KB][4] {f1, f2, X, 0}

    constexpr int TCOLS = NMAT == 2 ? 8 : 16;  // output columns per stage
    constexpr bool NORM = PRO == kProNorm;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int u0 = (int)((long long)p.n_units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)p.n_units * (blockIdx.x + 1) / gridDim.x);
    const int col_begin = u0 * p.unit;
    const int col_end = min(u1 * p.unit, p.N);
    if (col_begin >= col_end) return;  // uniform for the CTA, before any barrier
    const int ncols = col_end - col_begin;
    const int n_stages = (ncols + TCOLS - 1) / TCOLS;

    // =====================================================================
    // Producer warp.
    // =====================================================================
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            for (int s = 0; s < p.S; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kConsumerWarps);
                s_seq[s] = -1;
                s_cnt[s] = 0;
            }
            mbar_init(srows, 1);
            mbar_init(ready, 1);
            mbar_fence_init();
        }
        __syncwarp();
        lanes_bar_arrive(2, kThreads);
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            {
                // the CTA's scale and zero rows, one copy per array (the
                // range starts 16-byte aligned and G is a multiple of 4)
                const uint32_t bytes = (uint32_t)ncols * (uint32_t)p.G * 4u;
                mbar_arrive_expect_tx(srows, (uint32_t)NMAT * 2u * bytes);
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    bulk_g2s(smem + p.off_s[m], p.scales[m] + (size_t)col_begin * p.G, bytes, srows);
                    bulk_g2s(smem + p.off_z[m], p.zeros[m] + (size_t)col_begin * p.G, bytes, srows);
                }
            }
            for (int i = 0; ok && i < n_stages; ++i) {
                const int slot = i % p.S;
                // two stages go out at once, the rest after the consumers'
                // prologue (its activation loads are not queued behind the
                // whole ring's weight copies)
                if (i == 2 && !mbar_wait(ready, 0)) {
                    lanes_error();
                    ok = false;
                    break;
                }
                if (i >= p.S && !mbar_wait(&empty[slot], ((i / p.S) - 1) & 1)) {
                    lanes_error();
                    ok = false;
                    break;
                }
                const int c0 = col_begin + i * TCOLS;
                const int nc = min(TCOLS, col_end - c0);
                int rc[2], rn[2];  // first column and count of each region
                if constexpr (NMAT == 2) {
                    rc[0] = rc[1] = c0;
                    rn[0] = rn[1] = nc;
                } else {
                    rc[0] = c0;
                    rn[0] = min(8, nc);
                    rc[1] = c0 + 8;
                    rn[1] = nc - rn[0];
                }
                unsigned char *dst = smem + (size_t)slot * p.stage_bytes;
                s_seq[slot] = i;  // published by the release of the arrive below
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(rn[0] + rn[1]) * p.col_bytes);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (rn[r] == 0) continue;
                    const int m = NMAT == 2 ? r : 0;
                    bulk_g2s(dst + (r ? p.off_reg1 : 0u), p.Bq[m] + (size_t)rc[r] * (p.KW / 4),
                             (uint32_t)rn[r] * p.col_bytes, &full[slot]);
                }
                issued = i + 1;
            }
            if (!ok) {
                // leave no copy in flight into this CTA's shared memory
                (void)mbar_wait(srows, 0);
                for (int i = (issued > p.S ? issued - p.S : 0); i < issued; ++i)
                    (void)mbar_wait(&full[i % p.S], (i / p.S) & 1);
            }
        }
        return;
    }

    // =====================================================================
    // Consumer warps: prologue.  A thread takes the packed words w = base +
    // lane (+ kCT ...) of every lane m: their 8 activations, the block's scale
    // exponent and sum by shuffles over the 16 threads holding the block's 16
    // words, the fp16 high/low parts into the MMA's B layout.  All loads of a
    // batch of words are issued before any is used (one round trip per batch
    // under the weight stream); the loop bounds are uniform per warp, so the
    // shuffles always see all 32 lanes.
    // =====================================================================
    const int ctid = threadIdx.x;
    lanes_dependency_wait();
    float sq[NP];
#pragma unroll
    for (int m = 0; m < NP; ++m) sq[m] = 0.0f;
    const bool cta0 = blockIdx.x == 0;
    constexpr int WB = 2;                          // words per thread per batch
    constexpr bool TWO = PRO != kProNone;          // A_b (norm) or the gate vector
    const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int base = warp * 32; base < p.KW; base += kCT * WB) {
        float4 va[WB][NP][2], vb[WB][NP][2], vg[WB][2];
#pragma unroll
        for (int j = 0; j < WB; ++j) {
            const int w = base + lane + j * kCT;
            const bool ok = w < p.KW;
#pragma unroll
            for (int m = 0; m < NP; ++m) {
                const bool on = ok && m < p.M;
                const float4 *a4 = reinterpret_cast<const float4 *>(p.A + (size_t)m * p.K + (size_t)w * 8);
                va[j][m][0] = on ? __ldg(a4) : z4;
                va[j][m][1] = on ? __ldg(a4 + 1) : z4;
                if constexpr (TWO) {
                    const bool onb = on && p.A_b != nullptr;
                    const float4 *b4 = reinterpret_cast<const float4 *>(p.A_b + (size_t)m * p.K + (size_t)w * 8);
                    vb[j][m][0] = onb ? __ldg(b4) : z4;
                    vb[j][m][1] = onb ? __ldg(b4 + 1) : z4;
                }
            }
            if constexpr (NORM) {
                const float4 *g4 = reinterpret_cast<const float4 *>(p.W_norm + (size_t)w * 8);
                vg[j][0] = ok ? __ldg(g4) : z4;
                vg[j][1] = ok ? __ldg(g4 + 1) : z4;
            }
        }
#pragma unroll
        for (int j = 0; j < WB; ++j) {
            const int w = base + lane + j * kCT;
            const bool ok = w < p.KW;
#pragma unroll
            for (int m = 0; m < NP; ++m) {
                float4 v0 = va[j][m][0], v1 = va[j][m][1];
                if constexpr (NORM) {
                    const float4 b0 = vb[j][m][0], b1 = vb[j][m][1];
                    v0.x += b0.x; v0.y += b0.y; v0.z += b0.z; v0.w += b0.w;
                    v1.x += b1.x; v1.y += b1.y; v1.z += b1.z; v1.w += b1.w;
                    if (cta0 && ok && m < p.M && p.residual_out) {
                        float4 *r4 = reinterpret_cast<float4 *>(p.residual_out + (size_t)m * p.K + (size_t)w * 8);
                        r4[0] = v0;
                        r4[1] = v1;
                    }
                    float s2 = v0.x * v0.x;
                    s2 = fmaf(v0.y, v0.y, s2); s2 = fmaf(v0.z, v0.z, s2); s2 = fmaf(v0.w, v0.w, s2);
                    s2 = fmaf(v1.x, v1.x, s2); s2 = fmaf(v1.y, v1.y, s2);
                    s2 = fmaf(v1.z, v1.z, s2); s2 = fmaf(v1.w, v1.w, s2);
                    sq[m] += s2;
                    const float4 g0 = vg[j][0], g1 = vg[j][1];
                    v0.x *= g0.x; v0.y *= g0.y; v0.z *= g0.z; v0.w *= g0.w;
                    v1.x *= g1.x; v1.y *= g1.y; v1.z *= g1.z; v1.w *= g1.w;
                } else if constexpr (TWO) {
                    const float4 g0 = vb[j][m][0], g1 = vb[j][m][1];
                    v0.x = gate_input<PRO>(v0.x, g0.x); v0.y = gate_input<PRO>(v0.y, g0.y);
                    v0.z = gate_input<PRO>(v0.z, g0.z); v0.w = gate_input<PRO>(v0.w, g0.w);
                    v1.x = gate_input<PRO>(v1.x, g1.x); v1.y = gate_input<PRO>(v1.y, g1.y);
                    v1.z = gate_input<PRO>(v1.z, g1.z); v1.w = gate_input<PRO>(v1.w, g1.w);
                }
                const float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                stage_word<NP>(x, m, w, ok, lane, s_act, smem + p.off_fx);
            }
        }
    }
    if constexpr (NORM) {
        // inverse RMS per lane: xor tree in each warp, then warps in order
#pragma unroll
        for (int m = 0; m < NP; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sq[m] += __shfl_xor_sync(0xffffffffu, sq[m], off);
            if (lane == 0) s_sq[warp * 4 + m] = sq[m];
        }
        lanes_bar(1, kCT);
        if (ctid < NP) {
            float sum = 0.0f;
            for (int w = 0; w < kConsumerWarps; ++w) sum += s_sq[w * 4 + ctid];
            s_inv[ctid] = 1.0f / sqrtf(sum / (float)p.K + p.eps);
        }
    }
    lanes_bar(2, kThreads);  // activations staged; the producer has initialised the mbarriers
    if (ctid == 0) mbar_arrive(ready);

    // =====================================================================
    // Consumer warps: stages.
    // =====================================================================
    // `failed` stays uniform across each warp: the MMAs need every lane
    bool failed = !__all_sync(0xffffffffu, mbar_wait(srows, 0));
    if (failed) lanes_error();
    const int g = lane >> 2, t = lane & 3;
    // this warp's K slice: blocks [bw0, bw1), groups [gw0, gw1)
    const int bw0 = (int)((long long)p.KB * warp / kConsumerWarps);
    const int bw1 = (int)((long long)p.KB * (warp + 1) / kConsumerWarps);
    const int gw0 = bw0 / p.bpg;
    const int ngw = bw1 > bw0 ? (bw1 - 1) / p.bpg - gw0 + 1 : 0;
    float4 *scr = reinterpret_cast<float4 *>(smem + p.off_scr) + (size_t)warp * p.max_groups * 16;
    float2 *part = reinterpret_cast<float2 *>(smem + p.off_part);  // [S][warps][32]
    const float inv_t = NORM ? s_inv[t] : 1.0f;
    // MMA rows g and g + 8: region g & 1, columns (g >> 1) and (g >> 1) + 4 of it
    const uint32_t row_off = ((g & 1) ? p.off_reg1 : 0u) + (uint32_t)(g >> 1) * p.col_bytes;
    const uint32_t row8_delta = 4u * p.col_bytes;
    const uint32_t b_lane_off = (uint32_t)(g * 4 + t) * 16u;
    const bool b_active = g < 2 * NP;

    for (int i = 0; i < n_stages; ++i) {
        if (i == n_stages - 1 && lane == 0) lanes_dependents_launch();
        const int ring = i % p.S;
        const int c0 = col_begin + i * TCOLS;
        const int lc0 = i * TCOLS;  // CTA-relative first column of the stage
        if (!failed && !__all_sync(0xffffffffu, wait_shared_eq(&s_seq[ring], i) &&
                                                    mbar_wait(&full[ring], (i / p.S) & 1))) {
            lanes_error();
            failed = true;
        }
        const unsigned char *st = smem + (size_t)ring * p.stage_bytes;

        // scale and zero of this warp's groups for the tile's 16 MMA rows
        for (int idx = lane; idx < ngw * 16; idx += 32) {
            const int j = idx % ngw, r = idx / ngw;
            int m, lc;
            if constexpr (NMAT == 2) {
                m = r & 1;
                lc = lc0 + (r >> 1);
            } else {
                m = 0;
                lc = lc0 + 8 * (r & 1) + (r >> 1);
            }
            lc = lc < ncols ? lc : 0;  // past the range: any valid row (discarded)
            const size_t si = (size_t)lc * p.G + gw0 + j;
            const float* sr = reinterpret_cast<const float *>(smem + p.off_s[m]);
            const float* zr = reinterpret_cast<const float *>(smem + p.off_z[m]);
            // scale, fractional part of the zero, integer part as two fp16
            // subnormal halves (zi * 2^-24: the bit pattern zi)
            const float z = zr[si];
            const float zf = rintf(fminf(fmaxf(z, 0.0f), 15.0f));
            const uint32_t zbits = (uint32_t)(int)zf * 0x00010001u;
            scr[j * 16 + r] = make_float4(sr[si], z - zf, __uint_as_float(zbits), 0.0f);
        }
        __syncwarp();

        float y0 = 0.0f, y8 = 0.0f;
        if (!failed) {
            const unsigned char *ra = st + row_off;
            for (int b = bw0; b < bw1; ++b) {
                const uint4 wa = *reinterpret_cast<const uint4 *>(ra + b * 64 + t * 16);
                const uint4 wb = *reinterpret_cast<const uint4 *>(ra + row8_delta + b * 64 + t * 16);
                const int j = b / p.bpg - gw0;
                const float4 sz0 = scr[j * 16 + g];
                const float4 sz8 = scr[j * 16 + g + 8];
                // the integer zero, subtracted from the codes exactly: zi and
                // 16 zi as fp16 subnormals in both halves
                const uint32_t z0 = __float_as_uint(sz0.z), z8 = __float_as_uint(sz8.z);
                const uint32_t z0h = z0 << 4, z8h = z8 << 4;
                float d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                float d2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                const unsigned char *bb = s_act + (size_t)b * 4 * (2 * NP * 64) + b_lane_off;
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {
                    uint4 bq = make_uint4(0u, 0u, 0u, 0u);
                    if (b_active) bq = *reinterpret_cast<const uint4 *>(bb + pr * (2 * NP * 64));
                    const uint32_t w0 = pr == 0 ? wa.x : pr == 1 ? wa.y : pr == 2 ? wa.z : wa.w;
                    const uint32_t w8 = pr == 0 ? wb.x : pr == 1 ? wb.y : pr == 2 ? wb.z : wb.w;
                    mma_f16(d1, hsub2_bits(w0 & 0x000F000Fu, z0), hsub2_bits(w8 & 0x000F000Fu, z8),
                            hsub2_bits(w0 & 0x00F000F0u, z0h), hsub2_bits(w8 & 0x00F000F0u, z8h), bq.x, bq.y);
                    const uint32_t v0 = w0 >> 8, v8 = w8 >> 8;
                    mma_f16(d2, hsub2_bits(v0 & 0x000F000Fu, z0), hsub2_bits(v8 & 0x000F000Fu, z8),
                            hsub2_bits(v0 & 0x00F000F0u, z0h), hsub2_bits(v8 & 0x00F000F0u, z8h), bq.z, bq.w);
                }
                const float4 fx = s_fx[b * 4 + t];
                const float e0 = (d1[0] + d1[1]) + (d2[0] + d2[1]);
                const float e8 = (d1[2] + d1[3]) + (d2[2] + d2[3]);
                // y += s * (sum (q - zi) x - (z - zi) X)
                y0 = fmaf(sz0.x, fmaf(-sz0.y, fx.z, (e0 * fx.x) * fx.y), y0);
                y8 = fmaf(sz8.x, fmaf(-sz8.y, fx.z, (e8 * fx.x) * fx.y), y8);
            }
        }

        // ---- cross-warp sum: partials per ring entry, the last warp adds ----
        part[((size_t)ring * kConsumerWarps + warp) * 32 + lane] = make_float2(y0, y8);
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&s_cnt[ring], 1) == kConsumerWarps - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence_block();
            float a0 = 0.0f, a8 = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float2 v = part[((size_t)ring * kConsumerWarps + w) * 32 + lane];
                a0 += v.x;
                a8 += v.y;
            }
            a0 *= inv_t;
            a8 *= inv_t;
            if (failed) a0 = a8 = __int_as_float(0x7fffffff);
            const bool lane_ok = t < p.M;
            const int ci = g >> 1;  // column of row g within its region (row g + 8: ci + 4)
            if constexpr (EPI == kEpiGated) {
                // even g: gate rows; g + 1 (4 lanes on): the up rows of the same columns
                const float u0 = __shfl_down_sync(0xffffffffu, a0, 4);
                const float u8 = __shfl_down_sync(0xffffffffu, a8, 4);
                if ((g & 1) == 0 && lane_ok) {
                    const int ca = c0 + ci, cb = c0 + ci + 4;
                    if (ca < col_end) p.out[0][(size_t)t * p.N + ca] = a0 / (1.0f + expf(-a0)) * u0;
                    if (cb < col_end) p.out[0][(size_t)t * p.N + cb] = a8 / (1.0f + expf(-a8)) * u8;
                }
            } else if constexpr (EPI == kEpiDual) {
                if (lane_ok) {
                    float *o = p.out[g & 1];
                    const int ca = c0 + ci, cb = c0 + ci + 4;
                    if (ca < col_end) o[(size_t)t * p.N + ca] = a0;
                    if (cb < col_end) o[(size_t)t * p.N + cb] = a8;
                }
            } else {
                if (lane_ok) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int col = c0 + 8 * (g & 1) + ci + 4 * h;
                        if (col >= col_end) continue;
                        const float v = h ? a8 : a0;
                        if constexpr (EPI == kEpiQuad) {
                            const int seg = col < p.seg_start[1] ? 0 : col < p.seg_start[2] ? 1
                                          : col < p.seg_start[3] ? 2 : 3;
                            p.out[seg][(size_t)t * p.seg_len[seg] + (col - p.seg_start[seg])] = v;
                        } else {
                            p.out[0][(size_t)t * p.N + col] = v;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) s_cnt[ring] = 0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[ring]);  // after the sum: the partials stay until then
    }

    if constexpr (NORM) {
        // norm_out = (x * inv) * W_norm, written once (CTA 0)
        if (cta0 && p.norm_out) {
            const int K4 = p.K >> 2;
            for (int m = 0; m < p.M; ++m) {
                const size_t row = (size_t)m * p.K;
                const float inv = s_inv[m];
                for (int v4 = ctid; v4 < K4; v4 += kCT) {
                    float4 x = __ldg(reinterpret_cast<const float4 *>(p.A + row) + v4);
                    if (p.A_b) {
                        const float4 b = __ldg(reinterpret_cast<const float4 *>(p.A_b + row) + v4);
                        x.x += b.x; x.y += b.y; x.z += b.z; x.w += b.w;
                    }
                    const float4 gg = __ldg(reinterpret_cast<const float4 *>(p.W_norm) + v4);
                    x.x = (x.x * inv) * gg.x; x.y = (x.y * inv) * gg.y;
                    x.z = (x.z * inv) * gg.z; x.w = (x.w * inv) * gg.w;
                    reinterpret_cast<float4 *>(p.norm_out + row)[v4] = x;
                }
            }
        }
    }
}

template <int NMAT, int PRO, int EPI, int NP>
cudaError_t launch_lanes_variant(const LanesParams &prm, size_t smem, cudaStream_t stream)
{
    auto kern = lanes_matvec_kernel<NMAT, PRO, EPI, NP>;
    int dev = 0, sms = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    constexpr int kMaxDevices = 64;
    static std::atomic<unsigned char> smem_ready[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices || !smem_ready[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kSmemLimit + 4096u));
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   (int)cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < kMaxDevices) smem_ready[dev].store(1, std::memory_order_release);
    }
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    int grid = sms;
    if (grid > prm.n_units) grid = prm.n_units;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int NMAT, int PRO, int EPI>
cudaError_t launch_lanes_np(const LanesParams &prm, size_t smem, cudaStream_t stream)
{
    return prm.M <= 2 ? launch_lanes_variant<NMAT, PRO, EPI, 2>(prm, smem, stream)
                      : launch_lanes_variant<NMAT, PRO, EPI, 4>(prm, smem, stream);
}

int lanes_sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

// Shared-memory plan of a call; false when it does not fit this path.
bool plan_lanes(const Call &call, LanesParams &prm, size_t &smem, int grid)
{
    if (call.M < 2 || call.M > 4) return false;
    if (call.gs % kBlock != 0 || call.K % kBlock != 0 || call.K % call.gs != 0) return false;
    prm.M = call.M;
    prm.K = call.K;
    prm.N = call.N;
    prm.gs = call.gs;
    prm.KW = call.K / 8;
    prm.KB = call.K / kBlock;
    prm.G = call.K / call.gs;
    if (prm.G % 4 != 0) return false;  // every region's scale rows 16-byte aligned
    prm.bpg = call.gs / kBlock;
    prm.unit = 1;
    prm.n_units = call.N;
    if (grid > prm.n_units) grid = prm.n_units;
    const int max_cols = (prm.n_units + grid - 1) / grid;
    const int NP = call.M <= 2 ? 2 : 4;
    // the most groups a warp's slice of whole blocks touches
    int mg = 0;
    for (int w = 0; w < kConsumerWarps; ++w) {
        const int b0 = (int)((long long)prm.KB * w / kConsumerWarps);
        const int b1 = (int)((long long)prm.KB * (w + 1) / kConsumerWarps);
        const int n = (b1 - 1) / prm.bpg - b0 / prm.bpg + 1;
        if (b1 > b0 && n > mg) mg = n;
    }
    prm.max_groups = mg > 0 ? mg : 1;
    prm.col_bytes = (uint32_t)call.K / 2u;
    const uint32_t reg_bytes = 8u * prm.col_bytes;  // a multiple of 512
    prm.off_reg1 = reg_bytes + 64u;
    const uint32_t stage = round_up(prm.off_reg1 + reg_bytes, 128u);
    const uint32_t act_bytes = (uint32_t)prm.KB * 4u * (uint32_t)(2 * NP) * 64u;
    const uint32_t fx_bytes = (uint32_t)prm.KB * 4u * 16u;
    const uint32_t rows_bytes = round_up((uint32_t)max_cols * (uint32_t)prm.G * 4u, 128u);
    const uint32_t scr_bytes = round_up((uint32_t)kConsumerWarps * prm.max_groups * 16u * 16u, 128u);
    const uint32_t misc_bytes = 256u;
    const uint32_t bar_bytes = (2 * kMaxStages + 2) * 8u + 2 * kMaxStages * 4u;
    const uint32_t part_per_stage = (uint32_t)kConsumerWarps * 32u * 8u;
    const uint32_t fixed = act_bytes + fx_bytes + 2u * call.nmat * rows_bytes + scr_bytes + misc_bytes + bar_bytes;
    if (fixed + 2u * (stage + part_per_stage) > kSmemLimit) return false;
    int S = (int)((kSmemLimit - fixed) / (stage + part_per_stage));
    if (S > kMaxStages) S = kMaxStages;
    prm.S = S;
    prm.stage_bytes = stage;
    uint32_t off = round_up((uint32_t)S * stage, 128u);
    for (int m = 0; m < 2; ++m) {
        if (m < call.nmat) {
            prm.off_s[m] = off;
            off += rows_bytes;
            prm.off_z[m] = off;
            off += rows_bytes;
        } else {
            prm.off_s[m] = prm.off_s[0];
            prm.off_z[m] = prm.off_z[0];
        }
    }
    prm.off_act = off;
    off += act_bytes;
    prm.off_fx = off;
    off += fx_bytes;
    prm.off_part = off;
    off += round_up((uint32_t)S * part_per_stage, 128u);
    prm.off_scr = off;
    off += scr_bytes;
    prm.off_misc = off;
    off += misc_bytes;
    prm.off_bar = off;
    off += bar_bytes;
    smem = off;
    return smem <= kSmemLimit + 4096u;
}

}  // namespace

bool lanes_path_supported(const Call &call)
{
    if (call.M < 2 || call.M > 4) return false;
    for (int m = 0; m < call.nmat; ++m) {
        if ((reinterpret_cast<uintptr_t>(call.scales[m]) & 15u) != 0) return false;
        if ((reinterpret_cast<uintptr_t>(call.zeros[m]) & 15u) != 0) return false;
    }
    // the variants launch_lanes instantiates
    const int pro = prologue_of(call);
    const bool variant = call.epi == kEpiStore ||
                         (call.epi == kEpiQuad && pro == kProNone) ||
                         (call.epi == kEpiGated && (pro == kProNone || pro == kProNorm)) ||
                         (call.epi == kEpiDual && pro == kProNone);
    if (!variant) return false;
    LanesParams prm{};
    size_t smem;
    const int sms = lanes_sm_count();
    return sms > 0 && plan_lanes(call, prm, smem, sms);
}

cudaError_t launch_lanes(const Call &call, cudaStream_t stream)
{
    LanesParams prm{};
    size_t smem = 0;
    const int sms = lanes_sm_count();
    if (sms <= 0 || !plan_lanes(call, prm, smem, sms)) return cudaErrorInvalidValue;
    prm.A = call.A;
    if (call.norm) {
        prm.A_b = call.norm->A_b;
        prm.W_norm = call.norm->W_norm;
        prm.eps = call.norm->eps;
        prm.residual_out = call.norm->residual_out;
        prm.norm_out = call.norm->norm_out;
    } else if (call.gate_kind != kGateNone) {
        prm.A_b = call.G;  // the gate vector
    }
    for (int m = 0; m < 2; ++m) {
        const int src = m < call.nmat ? m : 0;
        prm.Bq[m] = reinterpret_cast<const uint4 *>(call.Bq[src]);
        prm.scales[m] = call.scales[src];
        prm.zeros[m] = call.zeros[src];
    }
    for (int i = 0; i < 4; ++i) {
        prm.out[i] = call.out[i];
        prm.seg_start[i] = call.seg_start[i];
        prm.seg_len[i] = call.seg_len[i];
    }
    const int pro = prologue_of(call);
    switch (call.epi) {
    case kEpiStore:
        switch (pro) {
        case kProNorm: return launch_lanes_np<1, kProNorm, kEpiStore>(prm, smem, stream);
        case kProSigmoid: return launch_lanes_np<1, kProSigmoid, kEpiStore>(prm, smem, stream);
        case kProSwiglu: return launch_lanes_np<1, kProSwiglu, kEpiStore>(prm, smem, stream);
        default: return launch_lanes_np<1, kProNone, kEpiStore>(prm, smem, stream);
        }
    case kEpiQuad:
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_lanes_np<1, kProNone, kEpiQuad>(prm, smem, stream);
    case kEpiGated:
        if (pro == kProNorm) return launch_lanes_np<2, kProNorm, kEpiGated>(prm, smem, stream);
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_lanes_np<2, kProNone, kEpiGated>(prm, smem, stream);
    case kEpiDual:
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_lanes_np<2, kProNone, kEpiDual>(prm, smem, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t read_lanes_device_error(unsigned int *bits, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(bits, g_lanes_error, sizeof(unsigned int));
    if (err != cudaSuccess || !clear) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_lanes_error, &zero, sizeof(unsigned int));
}

}  // namespace gq4

// gq4_quant.cu -- producing the int4 format on the GPU: the group-wise
// quantizer (gq4_quantize) and the MLX affine converter (gq4_from_mlx).
//
// Quantizer (the gpu bundle's loader quantizes the backbone's linears
// weight-only, group-wise to INT4: quantizeInt4 / quantizeBackboneInt4, whose
// body the pages do not show).  Per group of gs consecutive inputs of one
// column, a min/max asymmetric map onto the 16 codes with a float zero point;
// every step is one binary32 operation with round-to-nearest-even, so the
// codes are decided exactly as the header states:
//   lo, hi = min, max (+0.0: no negative zero); d = hi - lo
//   s = d / 15 (1 when below FLT_MIN); z = -lo / s; r = 1 / s
//   q = clamp(rint((v - lo) * r), 0, 15)
// A group with a non-finite value or an overflowing range gets codes 0 and a
// NaN scale and zero, and raises bit 3 of the device error word.
//
// MLX conversion (gpu bundle 1.0.0, dequantizeMLXProjection: the same word
// layout with w = scale * q + bias per group): zero = -bias / scale; a group
// without a finite zero (scale 0, or an overflowing quotient with a finite
// bias) becomes codes 1 with scale = bias and zero 0, which is w = bias.
//
// Both kernels are HBM-bound streams: the quantizer reads 4 bytes and writes
// 0.5 + 8/gs bytes per weight; the converter reads and writes 0.5 + 8/gs.
// Layout: a column's groups are contiguous, so group gi = n*G + g owns the
// gs floats of W and the gs/8 words of Bq starting at gi*gs and gi*gs/8.
#include <cfloat>
#include <cstdint>

#include "gq4_device.cuh"
#include "gq4_internal.h"

namespace gq4 {
namespace {

__device__ unsigned int g_quant_error = 0;
constexpr unsigned int kQuantNonFinite = 1u << 3;

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 2;  // warp tasks whose loads are issued together

struct QuantParams {
    const float4 *W;
    uint32_t *Bq;
    float *scales;
    float *zeros;
    long long n_groups;
    long long n_tasks;  // warp tasks
    int wpg;            // words per group (gs / 8)
    int L;              // lanes per group, min(wpg, 32)
    int P;              // groups per warp task
};

// min and max that return NaN when either input is NaN, so that a NaN
// anywhere in a group reaches its range.
__device__ __forceinline__ float min_nan(float a, float b)
{
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float max_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// min and max over the L consecutive lanes of this lane's segment (segments
// start at multiples of L, L <= 32).  A power of two: an xor butterfly that
// leaves the result in every lane.  Otherwise a tree towards the segment's
// first lane and a broadcast from it; lanes past the last whole segment
// only ever read themselves.
__device__ __forceinline__ void segment_min_max(float &lo, float &hi, int pos, int head, int L)
{
    if ((L & (L - 1)) == 0) {
        for (int off = L >> 1; off > 0; off >>= 1) {
            lo = min_nan(lo, __shfl_xor_sync(0xffffffffu, lo, off));
            hi = max_nan(hi, __shfl_xor_sync(0xffffffffu, hi, off));
        }
        return;
    }
    for (int off = 1; off < L; off <<= 1) {
        const float l2 = __shfl_down_sync(0xffffffffu, lo, off);
        const float h2 = __shfl_down_sync(0xffffffffu, hi, off);
        if (pos + off < L) {
            lo = min_nan(lo, l2);
            hi = max_nan(hi, h2);
        }
    }
    lo = __shfl_sync(0xffffffffu, lo, head);
    hi = __shfl_sync(0xffffffffu, hi, head);
}

__device__ __forceinline__ bool finite_f32(float v)
{
    return fabsf(v) <= FLT_MAX;  // false for NaN and +-inf
}

// Scale, zero and reciprocal of a group from its min and max (NaN when the
// group holds a NaN).  The group is bad when its range is not finite: a NaN,
// an infinity (inf - x, x - (-inf) or inf - inf) or an overflowing
// difference, exactly the groups the oracle rejects value by value.
struct GroupMap {
    float lo, s, r, z;
};

__device__ __forceinline__ GroupMap group_map(float lo, float hi, int &bad)
{
    GroupMap m;
    m.lo = __fadd_rn(lo, 0.0f);  // -0 becomes +0
    hi = __fadd_rn(hi, 0.0f);
    const float d = __fsub_rn(hi, m.lo);
    bad = finite_f32(d) ? 0 : 1;
    float s = __fdiv_rn(d, 15.0f);
    if (s < FLT_MIN) s = 1.0f;
    m.s = s;
    m.r = __frcp_rn(s);
    m.z = __fdiv_rn(-m.lo, s);
    return m;
}

// The 8 codes of one word: t = fl(fl(v - lo) * r) in packed pairs, then
// rounded to the nearest integer, ties to even, by cvt.rni.  (Rounding by
// adding 1.5 * 2^23 is not used: an add after the multiply may be fused into
// one FMA, which rounds the exact product instead of t.)  For a good group
// 0 <= t <= 15 (1 + 4u), so the code needs no clamp.  The eight codes are
// gathered by byte permutes into even and odd codes and merged as nibbles.
__device__ __forceinline__ uint32_t quantize_word(const float (&v)[8], const GroupMap &m)
{
    const f32x2 nlo = pack2(-m.lo, -m.lo), r = pack2(m.r, m.r);
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const float2 t = unpack2(mul2(add2(pack2(v[i], v[i + 1]), nlo), r));
        b[i] = (uint32_t)__float2int_rn(t.x);
        b[i + 1] = (uint32_t)__float2int_rn(t.y);
    }
    const uint32_t even = __byte_perm(__byte_perm(b[0], b[2], 0x0040),
                                      __byte_perm(b[4], b[6], 0x0040), 0x5410);
    const uint32_t odd = __byte_perm(__byte_perm(b[1], b[3], 0x0040),
                                     __byte_perm(b[5], b[7], 0x0040), 0x5410);
    return even | (odd << 4);
}

// One word's 8 weights; STREAM: read once (evict-first), else kept in cache
// for a second pass.
template <bool STREAM>
__device__ __forceinline__ void load_word(const float4 *W, long long word, float (&v)[8])
{
    const float4 a = STREAM ? __ldcs(W + 2 * word) : W[2 * word];
    const float4 b = STREAM ? __ldcs(W + 2 * word + 1) : W[2 * word + 1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store_group_params(const QuantParams &p, long long gi, GroupMap m,
                                                   int bad)
{
    if (bad) {
        p.scales[gi] = __int_as_float(0x7fc00000);
        p.zeros[gi] = __int_as_float(0x7fc00000);
        atomicOr(&g_quant_error, kQuantNonFinite);
    } else {
        p.scales[gi] = m.s;
        p.zeros[gi] = m.z;
    }
}

// Groups of at most 32 words: P = 32 / L groups per warp task, one word
// (8 weights, two float4) per lane, a task covering P*L consecutive words.
__global__ void __launch_bounds__(kQuantThreads) quantize_narrow_kernel(QuantParams p)
{
    const int lane = threadIdx.x & 31;
    const int slot = lane / p.L;
    const int pos = lane - slot * p.L;
    const int head = lane - pos;
    const long long warp0 = ((long long)blockIdx.x * kQuantThreads + threadIdx.x) >> 5;
    const long long n_warps = ((long long)gridDim.x * kQuantThreads) >> 5;
    for (long long t0 = warp0; t0 < p.n_tasks; t0 += n_warps * kQuantUnroll) {
        float v[kQuantUnroll][8];
        long long gi[kQuantUnroll];
        bool active[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const long long task = t0 + (long long)u * n_warps;
            gi[u] = task * p.P + slot;
            active[u] = task < p.n_tasks && slot < p.P && gi[u] < p.n_groups;
            if (active[u]) {
                load_word<true>(p.W, gi[u] * p.wpg + pos, v[u]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[u][i] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            // warp-uniform: the whole warp takes part in the shuffles
            if (t0 + (long long)u * n_warps >= p.n_tasks) break;
            float lo = v[u][0], hi = v[u][0];
#pragma unroll
            for (int i = 1; i < 8; ++i) {
                lo = min_nan(lo, v[u][i]);
                hi = max_nan(hi, v[u][i]);
            }
            segment_min_max(lo, hi, pos, head, p.L);
            int bad;
            const GroupMap m = group_map(lo, hi, bad);
            if (!active[u]) continue;
            p.Bq[gi[u] * p.wpg + pos] = bad ? 0u : quantize_word(v[u], m);
            if (pos == 0) store_group_params(p, gi[u], m, bad);
        }
    }
    // The matvec kernels may start streaming these weights as soon as this
    // grid's blocks have exited (programmatic dependent launch, before their
    // dependency wait): make every store visible GPU-wide before exit.
    __threadfence();
}

// Groups of more than 32 words: one warp per group, lanes striding over its
// words; a first pass for min and max, a second (re-reading the group) for
// the codes.
__global__ void __launch_bounds__(kQuantThreads) quantize_wide_kernel(QuantParams p)
{
    const int lane = threadIdx.x & 31;
    const long long warp0 = ((long long)blockIdx.x * kQuantThreads + threadIdx.x) >> 5;
    const long long n_warps = ((long long)gridDim.x * kQuantThreads) >> 5;
    for (long long gi = warp0; gi < p.n_groups; gi += n_warps) {
        const long long w0 = gi * p.wpg;
        float lo = FLT_MAX, hi = -FLT_MAX;  // every lane has a word (wpg > 32)
        for (int j = lane; j < p.wpg; j += 32) {
            float v[8];
            load_word<false>(p.W, w0 + j, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lo = min_nan(lo, v[i]);
                hi = max_nan(hi, v[i]);
            }
        }
        segment_min_max(lo, hi, lane, 0, 32);
        int bad;
        const GroupMap m = group_map(lo, hi, bad);
        for (int j = lane; j < p.wpg; j += 32) {
            uint32_t word = 0u;
            if (!bad) {
                float v[8];
                load_word<false>(p.W, w0 + j, v);
                word = quantize_word(v, m);
            }
            p.Bq[w0 + j] = word;
        }
        if (lane == 0) store_group_params(p, gi, m, bad);
    }
    // The matvec kernels may start streaming these weights as soon as this
    // grid's blocks have exited (programmatic dependent launch, before their
    // dependency wait): make every store visible GPU-wide before exit.
    __threadfence();
}

// MLX conversion: one thread per 4 words (32 codes, always inside one
// group since a group holds a multiple of 4 words), grid-stride.  In place
// (Bq == packed) only the rewritten groups' words are stored.
constexpr int kMlxUnroll = 4;  // chunks per thread whose loads are issued together

__global__ void __launch_bounds__(256) from_mlx_kernel(long long n_chunks, int wpg,
                                                      const uint4 *packed,
                                                      const float *__restrict__ mlx_scales,
                                                      const float *__restrict__ mlx_biases,
                                                      uint4 *Bq, float *scales, float *zeros,
                                                      int in_place)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long c0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; c0 < n_chunks;
         c0 += stride * kMlxUnroll) {
        uint4 w[kMlxUnroll];
        float s[kMlxUnroll], b[kMlxUnroll];
#pragma unroll
        for (int u = 0; u < kMlxUnroll; ++u) {
            const long long c = c0 + u * stride;
            if (c < n_chunks) {
                const long long gi = 4 * c / wpg;
                s[u] = mlx_scales[gi];
                b[u] = mlx_biases[gi];
                if (!in_place) w[u] = __ldcs(packed + c);
            }
        }
#pragma unroll
        for (int u = 0; u < kMlxUnroll; ++u) {
            const long long c = c0 + u * stride;
            if (c >= n_chunks) break;
            const long long word = 4 * c;
            const long long gi = word / wpg;
            const float z = __fdiv_rn(-b[u], s[u]);
            const bool degenerate = s[u] == 0.0f || (isinf(z) && finite_f32(b[u]));
            if (degenerate) {
                __stcs(Bq + c, make_uint4(0x11111111u, 0x11111111u, 0x11111111u, 0x11111111u));
            } else if (!in_place) {
                __stcs(Bq + c, w[u]);
            }
            if (word == gi * wpg) {
                scales[gi] = degenerate ? b[u] : s[u];
                zeros[gi] = degenerate ? 0.0f : z;
            }
        }
    }
    // visible GPU-wide before exit: a following matvec may stream these
    // weights before its dependency wait (programmatic dependent launch)
    __threadfence();
}

int resident_blocks(const void *kernel)
{
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, kQuantThreads, 0) !=
        cudaSuccess)
        return 1;
    return blocks > 0 ? blocks : 1;
}

}  // namespace

cudaError_t launch_quantize(int K, int N, int gs, const float *W, uint32_t *Bq, float *scales,
                            float *zeros, cudaStream_t stream)
{
    static const int narrow_blocks = resident_blocks((const void *)quantize_narrow_kernel);
    static const int wide_blocks = resident_blocks((const void *)quantize_wide_kernel);
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    QuantParams p{};
    p.W = reinterpret_cast<const float4 *>(W);
    p.Bq = Bq;
    p.scales = scales;
    p.zeros = zeros;
    p.n_groups = (long long)N * (long long)(K / gs);
    p.wpg = gs / 8;
    const long long warps_per_block = kQuantThreads / 32;
    if (p.wpg <= 32) {
        p.L = p.wpg;
        p.P = 32 / p.L;
        p.n_tasks = (p.n_groups + p.P - 1) / p.P;
        const long long want = (p.n_tasks + warps_per_block * kQuantUnroll - 1) /
                               (warps_per_block * kQuantUnroll);
        const long long cap = (long long)sms * narrow_blocks;
        const unsigned grid = (unsigned)(want < cap ? want : cap);
        quantize_narrow_kernel<<<grid, kQuantThreads, 0, stream>>>(p);
    } else {
        p.L = 32;
        p.P = 1;
        p.n_tasks = p.n_groups;
        const long long want = (p.n_groups + warps_per_block - 1) / warps_per_block;
        const long long cap = (long long)sms * wide_blocks;
        const unsigned grid = (unsigned)(want < cap ? want : cap);
        quantize_wide_kernel<<<grid, kQuantThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_from_mlx(int K, int N, int gs, const uint32_t *packed, const float *mlx_scales,
                            const float *mlx_biases, uint32_t *Bq, float *scales, float *zeros,
                            cudaStream_t stream)
{
    static const int mlx_blocks = [] {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, from_mlx_kernel, 256, 0) !=
            cudaSuccess)
            return 1;
        return b > 0 ? b : 1;
    }();
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const long long n_chunks = (long long)N * (long long)(K / 32);
    const long long want = (n_chunks + 256 * kMlxUnroll - 1) / (256 * kMlxUnroll);
    const long long cap = (long long)sms * mlx_blocks;
    const unsigned blocks = (unsigned)(want < cap ? want : cap);
    from_mlx_kernel<<<blocks, 256, 0, stream>>>(
        n_chunks, gs / 8, reinterpret_cast<const uint4 *>(packed), mlx_scales, mlx_biases,
        reinterpret_cast<uint4 *>(Bq), scales, zeros, packed == Bq ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t read_quant_device_error(unsigned int *bits, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(bits, g_quant_error, sizeof(unsigned int));
    if (err != cudaSuccess || !clear) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(unsigned int));
}

}  // namespace gq4

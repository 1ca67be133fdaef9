// gq4_fp32.cu -- CUDA-core fp32 kernels for the int4 group-quantized matvec
// family: plain matvec, quad-output routing, RMSNorm prologue and SiLU-gated
// gate/up, for 1 <= M <= 32 decode lanes.
//
// Operation (gerbil moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 and
// WGSL_NORM_MATVEC_INT4; the DualMatVecInt4, GatedMatVecInt4 and
// SwiGLUGatedMatVecInt4 fusion docs): C[m][n] = sum_k a[m][k] * (q(n,k) - z)
// * s, with the code layout and dequant rule described in gq4.h.
//
// Work decomposition (GB300-first; the WGSL 16 x 16 workgroup is not kept):
//   * CTA = 8 warps.  grid.x walks lane blocks of MB lanes (fastest, so the
//     lane blocks that share a column tile run together and hit L2), grid.y
//     walks column tiles of 16 columns (2 weight streams per warp: two
//     columns, or the gate and up column of one output for the gated call).
//   * The CTA stages its lanes' activations for a K tile in shared memory,
//     pre-scaled by 16^-p (see gq4_device.cuh) and XOR-swizzled so that the
//     32 lanes of a warp, each reading a different 32-element chunk, hit
//     distinct banks.  The norm prologue (x = A + A_b, inverse RMS, gain) is
//     applied while staging, once per CTA; CTAs of column tile 0 also write
//     residual_out and norm_out.
//   * Lane l of a warp owns chunks c = l, l + 32, ... of every column: one
//     coalesced 128-bit load per column per chunk (a warp reads 512
//     contiguous bytes of a column), software-pipelined one chunk ahead.
//   * Per chunk: codes are unpacked in registers, (q - z) formed exactly, an
//     f32x2 FMA chain accumulates a * (q - z) over the 32 codes, and the
//     group scale multiplies the chunk sum (a chunk never straddles a group).
//   * Partial sums are reduced across the warp with a fixed xor butterfly,
//     so results are deterministic and independent of where a column sits in
//     a tile (quad == plain, lane == solo, bit for bit).
#include <atomic>
#include <cstdint>

#include "gq4_device.cuh"
#include "gq4_internal.h"

namespace gq4 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStreams = 2;                 // weight streams per warp
// Activation tile, bytes: dynamic shared memory plus the kernel's static
// arrays must stay within the 48 KB a launch gets without opting in.
constexpr int kSmemBudget = 47 * 1024;
// A whole-K activation tile may take up to this much (opt-in above 48 KB):
// two CTAs still fit on an SM.
constexpr size_t kSmemSingleMax = 100 * 1024;

struct Fp32Params {
    int M, K, N, gs;
    int KC;           // 32-code chunks per column (K / 32)
    int G;            // groups per column (K / gs)
    int kct;          // chunks per staged K tile
    int n_ktiles;
    int col_tiles;    // tiles of columns; a CTA takes blockIdx.y, + gridDim.y, ...
    unsigned long long group_magic;  // ceil(2^40 / (gs / 32))
    uint32_t magic_bits;             // kMagicBits, read from the parameter bank
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

__device__ __forceinline__ int chunk_group(int gc, unsigned long long magic)
{
    // floor(gc / (gs/32)) for gc < 2^20 (exact by the choice of magic).
    return (int)(((unsigned long long)gc * magic) >> 40);
}

__device__ __forceinline__ float4 prescale(float4 v)
{
    // float4 j of a chunk covers codes 0..3 (j even) or 4..7 (j odd) of word
    // j/2; both halves sit at code positions p = 0, 1, 2, 3.
    v.x *= code_prescale(0);
    v.y *= code_prescale(1);
    v.z *= code_prescale(2);
    v.w *= code_prescale(3);
    return v;
}

// One element of a gated input: x * sigmoid(g) or silu(g) * x (the same
// formulas as the one-lane kernel's prologue).
template <int PRO>
__device__ __forceinline__ float gate_input(float x, float g)
{
    if constexpr (PRO == kProSigmoid)
        return x / (1.0f + expf(-g));
    else
        return g / (1.0f + expf(-g)) * x;
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return g / (1.0f + expf(-g)) * u;
}

template <int MB, int NMAT, int PRO, int EPI>
__global__ void __launch_bounds__(kThreads)
fp32_matvec_kernel(const __grid_constant__ Fp32Params p)
{
    extern __shared__ __align__(16) float4 s_act[];   // [MB][kct][8], swizzled
    __shared__ float s_part[kWarps][MB];
    __shared__ float s_inv[MB];

    constexpr int CW = kStreams / NMAT;               // columns per warp
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int m0 = blockIdx.x * MB;
    const int nb = min(MB, p.M - m0);
    // RMSNorm: the inverse RMS is a per-lane scalar, so it is taken out of
    // the dot product: the staged activations are x * W_norm (x = A + A_b),
    // the square sum of x is accumulated while staging (each CTA stages all
    // of K), and the finished sums are scaled by 1/sqrt(sum/K + eps).  Each
    // lane's elements go to threads in a fixed order independent of MB, so a
    // lane's result does not depend on the lane count.
    float sq[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) sq[m] = 0.0f;
    constexpr bool NORM = PRO == kProNorm;
    const bool write_norm_outputs = NORM && blockIdx.y == 0;

    // Column tiles blockIdx.y, + gridDim.y, ...  With a single K tile the
    // activations are staged once and serve every column tile of the CTA
    // (the grid is then sized to the resident CTAs); otherwise each CTA
    // takes one column tile and stages K tile by tile.
    for (int tile = blockIdx.y; tile < p.col_tiles; tile += gridDim.y) {
    const bool first_tile = tile == (int)blockIdx.y;
    const int col_base = (tile * kWarps + warp) * CW;

    // ---- the warp's two weight streams ----
    const uint4 *wp[kStreams];
    const float *sp[kStreams];
    const float *zp[kStreams];
    bool valid[kStreams];
    int col[kStreams];
#pragma unroll
    for (int s = 0; s < kStreams; ++s) {
        const int mat = NMAT == 2 ? s : 0;
        col[s] = NMAT == 2 ? col_base : col_base + s;
        valid[s] = col[s] < p.N;
        const int c = valid[s] ? col[s] : 0;
        wp[s] = p.Bq[mat] + (size_t)c * p.KC;
        sp[s] = p.scales[mat] + (size_t)c * p.G;
        zp[s] = p.zeros[mat] + (size_t)c * p.G;
    }

    float acc[MB][kStreams];
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int s = 0; s < kStreams; ++s) acc[m][s] = 0.0f;

    for (int t = 0; t < p.n_ktiles; ++t) {
        const int kc0 = t * p.kct;
        const int kcn = min(p.kct, p.KC - kc0);
        if (first_tile || p.n_ktiles > 1) {
        __syncthreads();  // previous tile consumed
        // ---- stage activations of this K tile ----
        const int per_lane = kcn * 8;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            for (int r = tid; r < per_lane; r += kThreads) {
                const int c = r >> 3;
                const int j = r & 7;
                const size_t k = (size_t)(kc0 + c) * 32 + (size_t)j * 4;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (m < nb) {
                    const size_t row = (size_t)(m0 + m) * p.K;
                    v = *reinterpret_cast<const float4 *>(p.A + row + k);
                    if constexpr (NORM) {
                        if (p.A_b) {
                            const float4 b = *reinterpret_cast<const float4 *>(p.A_b + row + k);
                            v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
                        }
                        if (write_norm_outputs && p.residual_out)
                            *reinterpret_cast<float4 *>(p.residual_out + row + k) = v;
                        sq[m] = fmaf(v.x, v.x, sq[m]);
                        sq[m] = fmaf(v.y, v.y, sq[m]);
                        sq[m] = fmaf(v.z, v.z, sq[m]);
                        sq[m] = fmaf(v.w, v.w, sq[m]);
                        const float4 g = *reinterpret_cast<const float4 *>(p.W_norm + k);
                        v.x *= g.x; v.y *= g.y; v.z *= g.z; v.w *= g.w;
                    } else if constexpr (PRO != kProNone) {
                        // the gated input: x * sigmoid(g), or silu(g) * x
                        const float4 g = *reinterpret_cast<const float4 *>(p.A_b + row + k);
                        v.x = gate_input<PRO>(v.x, g.x);
                        v.y = gate_input<PRO>(v.y, g.y);
                        v.z = gate_input<PRO>(v.z, g.z);
                        v.w = gate_input<PRO>(v.w, g.w);
                    }
                }
                s_act[((size_t)m * p.kct + c) * 8 + (j ^ (c & 7))] = prescale(v);
            }
        }
        __syncthreads();
        }

        // ---- main loop: lane owns chunks lane, lane + 32, ... ----
        int c = lane;
        uint4 wq[kStreams];
        float sc[kStreams], zr[kStreams];
        if (c < kcn) {
            const int gc = kc0 + c;
            const int g = chunk_group(gc, p.group_magic);
#pragma unroll
            for (int s = 0; s < kStreams; ++s) {
                wq[s] = valid[s] ? __ldg(wp[s] + gc) : make_uint4(0u, 0u, 0u, 0u);
                sc[s] = valid[s] ? __ldg(sp[s] + g) : 0.0f;
                zr[s] = valid[s] ? __ldg(zp[s] + g) : 0.0f;
            }
        }
        for (; c < kcn; c += 32) {
            // prefetch the next chunk of both streams
            uint4 nwq[kStreams];
            float nsc[kStreams], nzr[kStreams];
            const int cn = c + 32;
            if (cn < kcn) {
                const int gc = kc0 + cn;
                const int g = chunk_group(gc, p.group_magic);
#pragma unroll
                for (int s = 0; s < kStreams; ++s) {
                    nwq[s] = valid[s] ? __ldg(wp[s] + gc) : make_uint4(0u, 0u, 0u, 0u);
                    nsc[s] = valid[s] ? __ldg(sp[s] + g) : 0.0f;
                    nzr[s] = valid[s] ? __ldg(zp[s] + g) : 0.0f;
                }
            }

            ZeroPairs zps[kStreams];
#pragma unroll
            for (int s = 0; s < kStreams; ++s) zps[s] = scaled_zero(zr[s]);

            f32x2 inner[MB][kStreams];
#pragma unroll
            for (int m = 0; m < MB; ++m)
#pragma unroll
                for (int s = 0; s < kStreams; ++s) inner[m][s] = 0ull;

            const ulonglong2 *arow = reinterpret_cast<const ulonglong2 *>(s_act);
            const f32x2 nmagic2 = neg_magic2();
            const int sw = c & 7;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                DiffPairs d[kStreams];
#pragma unroll
                for (int s = 0; s < kStreams; ++s) {
                    const uint32_t word = w == 0 ? wq[s].x : w == 1 ? wq[s].y : w == 2 ? wq[s].z : wq[s].w;
                    d[s] = code_minus_zero(word, zps[s], nmagic2, p.magic_bits);
                }
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    const size_t base = ((size_t)m * p.kct + c) * 8;
                    const ulonglong2 lo = arow[base + ((2 * w) ^ sw)];
                    const ulonglong2 hi = arow[base + ((2 * w + 1) ^ sw)];
#pragma unroll
                    for (int s = 0; s < kStreams; ++s) {
                        f32x2 a = inner[m][s];
                        a = fma2(lo.x, d[s].d01, a);
                        a = fma2(lo.y, d[s].d23, a);
                        a = fma2(hi.x, d[s].d45, a);
                        a = fma2(hi.y, d[s].d67, a);
                        inner[m][s] = a;
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MB; ++m)
#pragma unroll
                for (int s = 0; s < kStreams; ++s) {
                    const float2 v = unpack2(inner[m][s]);
                    acc[m][s] = fmaf(sc[s], v.x + v.y, acc[m][s]);
                }

#pragma unroll
            for (int s = 0; s < kStreams; ++s) {
                wq[s] = nwq[s];
                sc[s] = nsc[s];
                zr[s] = nzr[s];
            }
        }
    }

    if constexpr (NORM) {
        // inverse RMS per lane (once): fixed xor tree within each warp, warps in order
        if (first_tile) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sq[m] += __shfl_xor_sync(0xffffffffu, sq[m], off);
            if (lane == 0) s_part[warp][m] = sq[m];
        }
        __syncthreads();
        if (tid < MB) {
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sum += s_part[w][tid];
            s_inv[tid] = 1.0f / sqrtf(sum / (float)p.K + p.eps);
        }
        __syncthreads();
        }
#pragma unroll
        for (int m = 0; m < MB; ++m)
#pragma unroll
            for (int s = 0; s < kStreams; ++s) acc[m][s] *= s_inv[m];
        // norm_out = (x * inv) * W_norm, written once (column tile 0)
        if (write_norm_outputs && first_tile && p.norm_out) {
            const int K4 = p.K >> 2;
            for (int m = 0; m < nb; ++m) {
                const size_t row = (size_t)(m0 + m) * p.K;
                const float inv = s_inv[m];
                for (int v4 = tid; v4 < K4; v4 += kThreads) {
                    float4 x = reinterpret_cast<const float4 *>(p.A + row)[v4];
                    if (p.A_b) {
                        const float4 b = reinterpret_cast<const float4 *>(p.A_b + row)[v4];
                        x.x += b.x; x.y += b.y; x.z += b.z; x.w += b.w;
                    }
                    const float4 g = reinterpret_cast<const float4 *>(p.W_norm)[v4];
                    x.x = (x.x * inv) * g.x; x.y = (x.y * inv) * g.y;
                    x.z = (x.z * inv) * g.z; x.w = (x.w * inv) * g.w;
                    reinterpret_cast<float4 *>(p.norm_out + row)[v4] = x;
                }
            }
        }
    }

    // ---- warp reduction (fixed butterfly) and epilogue ----
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int s = 0; s < kStreams; ++s)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                acc[m][s] += __shfl_xor_sync(0xffffffffu, acc[m][s], off);

    if (lane == 0) {
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        if (m >= nb) break;
        const size_t mm = (size_t)(m0 + m);
        if constexpr (EPI == kEpiGated) {
            if (valid[0]) p.out[0][mm * p.N + col[0]] = silu_mul(acc[m][0], acc[m][1]);
        } else if constexpr (EPI == kEpiDual) {
            // stream 0: the column of matrix 0, stream 1: the same column of matrix 1
            if (valid[0]) {
                p.out[0][mm * p.N + col[0]] = acc[m][0];
                p.out[1][mm * p.N + col[0]] = acc[m][1];
            }
        } else {
#pragma unroll
            for (int s = 0; s < kStreams; ++s) {
                if (!valid[s]) continue;
                const int cc = col[s];
                if constexpr (EPI == kEpiQuad) {
                    const int seg = cc < p.seg_start[1] ? 0 : cc < p.seg_start[2] ? 1
                                  : cc < p.seg_start[3] ? 2 : 3;
                    p.out[seg][mm * p.seg_len[seg] + (cc - p.seg_start[seg])] = acc[m][s];
                } else {
                    p.out[0][mm * p.N + cc] = acc[m][s];
                }
            }
        }
    }
    }  // lane 0
    }  // column tiles
}

template <int MB, int NMAT, int PRO, int EPI>
cudaError_t launch_variant(Fp32Params prm, cudaStream_t stream)
{
    auto kern = fp32_matvec_kernel<MB, NMAT, PRO, EPI>;
    const int lane_blocks = (prm.M + MB - 1) / MB;
    const int cols_per_cta = kWarps * (kStreams / NMAT);
    prm.col_tiles = (prm.N + cols_per_cta - 1) / cols_per_cta;
    if (prm.col_tiles > 65535) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)MB * prm.kct * 8 * sizeof(float4);
    int grid_y = prm.col_tiles;
    cudaError_t err;
    if (smem > (size_t)kSmemBudget) {
        // one K tile beyond the default 48 KB: opt in once per device
        int dev = 0;
        if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
        constexpr int kMaxDevices = 64;
        static std::atomic<unsigned char> ready[kMaxDevices];
        if (dev < 0 || dev >= kMaxDevices || !ready[dev].load(std::memory_order_acquire)) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemSingleMax);
            if (err != cudaSuccess) return err;
            if (dev >= 0 && dev < kMaxDevices) ready[dev].store(1, std::memory_order_release);
        }
    }
    if (prm.n_ktiles == 1) {
        // activations staged once per CTA: as many CTAs as are resident
        int dev = 0, sms = 0, per_sm = 0;
        if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) != cudaSuccess)
            return err;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        const int resident = (sms * per_sm + lane_blocks - 1) / lane_blocks;
        if (grid_y > resident) grid_y = resident;
    }
    dim3 grid(lane_blocks, grid_y);
    kern<<<grid, kThreads, smem, stream>>>(prm);
    return cudaGetLastError();
}

template <int MB>
cudaError_t dispatch_mb(const Call &call, const Fp32Params &prm, cudaStream_t stream)
{
    const int pro = prologue_of(call);
    switch (call.epi) {
    case kEpiStore:
        switch (pro) {
        case kProNorm: return launch_variant<MB, 1, kProNorm, kEpiStore>(prm, stream);
        case kProSigmoid: return launch_variant<MB, 1, kProSigmoid, kEpiStore>(prm, stream);
        case kProSwiglu: return launch_variant<MB, 1, kProSwiglu, kEpiStore>(prm, stream);
        default: return launch_variant<MB, 1, kProNone, kEpiStore>(prm, stream);
        }
    case kEpiQuad:
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_variant<MB, 1, kProNone, kEpiQuad>(prm, stream);
    case kEpiGated:
        if (pro == kProNorm) return launch_variant<MB, 2, kProNorm, kEpiGated>(prm, stream);
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_variant<MB, 2, kProNone, kEpiGated>(prm, stream);
    case kEpiDual:
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_variant<MB, 2, kProNone, kEpiDual>(prm, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_fp32(const Call &call, cudaStream_t stream)
{
    Fp32Params prm{};
    prm.M = call.M;
    prm.K = call.K;
    prm.N = call.N;
    prm.gs = call.gs;
    prm.KC = call.K / 32;
    prm.G = call.K / call.gs;
    const unsigned long long cpg = (unsigned long long)(call.gs / 32);
    prm.group_magic = ((1ull << 40) + cpg - 1) / cpg;
    prm.magic_bits = kMagicBits;
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
    for (int i = 0; i < 2; ++i) {
        const int src = i < call.nmat ? i : 0;
        prm.Bq[i] = reinterpret_cast<const uint4 *>(call.Bq[src]);
        prm.scales[i] = call.scales[src];
        prm.zeros[i] = call.zeros[src];
    }
    for (int i = 0; i < 4; ++i) {
        prm.out[i] = call.out[i];
        prm.seg_start[i] = call.seg_start[i];
        prm.seg_len[i] = call.seg_len[i];
    }

    const int MB = call.M == 1 ? 1 : call.M == 2 ? 2 : call.M <= 4 ? 4 : 8;
    // All of K in one tile when it fits kSmemSingleMax (the CTAs then stage
    // once and loop over column tiles); otherwise K tiles of a multiple of 32
    // chunks within the default 48 KB, so lane l owns chunks l, l+32, ... in
    // increasing order whatever the tiling (results independent of MB).
    const size_t whole = (size_t)MB * prm.KC * 8 * sizeof(float4);
    if (whole <= kSmemSingleMax) {
        prm.kct = prm.KC;
    } else {
        const int kct_max = kSmemBudget / (MB * 8 * (int)sizeof(float4)) / 32 * 32;
        prm.kct = prm.KC < kct_max ? prm.KC : kct_max;
    }
    prm.n_ktiles = (prm.KC + prm.kct - 1) / prm.kct;

    switch (MB) {
    case 1: return dispatch_mb<1>(call, prm, stream);
    case 2: return dispatch_mb<2>(call, prm, stream);
    case 4: return dispatch_mb<4>(call, prm, stream);
    default: return dispatch_mb<8>(call, prm, stream);
    }
}

// ---------------------------------------------------------------------------
// Test kernels: integer unpack and binary32 dequant through the same
// in-register extraction as the matvec kernels.
// ---------------------------------------------------------------------------
namespace {

__global__ void unpack_kernel(size_t words, const uint32_t *__restrict__ Bq, uint8_t *__restrict__ q,
                              uint32_t magic_bits)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= words) return;
    const CodePairs c = extract_word(Bq[i], magic_bits);
    const f32x2 nmagic2 = neg_magic2();
    const float2 v01 = unpack2(add2(c.p01, nmagic2));
    const float2 v23 = unpack2(add2(c.p23, nmagic2));
    const float2 v45 = unpack2(add2(c.p45, nmagic2));
    const float2 v67 = unpack2(add2(c.p67, nmagic2));
    // undo the position scale 16^p (exact) and convert the small integers
    const uint32_t q0 = (uint32_t)(v01.x * code_prescale(0));
    const uint32_t q1 = (uint32_t)(v01.y * code_prescale(1));
    const uint32_t q2 = (uint32_t)(v23.x * code_prescale(2));
    const uint32_t q3 = (uint32_t)(v23.y * code_prescale(3));
    const uint32_t q4 = (uint32_t)(v45.x * code_prescale(4));
    const uint32_t q5 = (uint32_t)(v45.y * code_prescale(5));
    const uint32_t q6 = (uint32_t)(v67.x * code_prescale(6));
    const uint32_t q7 = (uint32_t)(v67.y * code_prescale(7));
    uint32_t *dst = reinterpret_cast<uint32_t *>(q + i * 8);
    dst[0] = q0 | (q1 << 8) | (q2 << 16) | (q3 << 24);
    dst[1] = q4 | (q5 << 8) | (q6 << 16) | (q7 << 24);
}

__global__ void dequant_kernel(size_t words, int K, int gs, const uint32_t *__restrict__ Bq,
                               const float *__restrict__ scales, const float *__restrict__ zeros,
                               float *__restrict__ W, uint32_t magic_bits)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= words) return;
    const size_t wpc = (size_t)(K / 8);
    const size_t n = i / wpc;
    const int k0 = (int)(i - n * wpc) * 8;
    const size_t g = n * (size_t)(K / gs) + (size_t)(k0 / gs);
    const float s = scales[g];
    const DiffPairs d = code_minus_zero(Bq[i], scaled_zero(zeros[g]), neg_magic2(), magic_bits);
    const float2 d01 = unpack2(d.d01), d23 = unpack2(d.d23), d45 = unpack2(d.d45), d67 = unpack2(d.d67);
    // d = 16^p * fl(q - zero): scale back exactly, then one rounding for * scale
    float *dst = W + i * 8;
    dst[0] = __fmul_rn(d01.x * code_prescale(0), s);
    dst[1] = __fmul_rn(d01.y * code_prescale(1), s);
    dst[2] = __fmul_rn(d23.x * code_prescale(2), s);
    dst[3] = __fmul_rn(d23.y * code_prescale(3), s);
    dst[4] = __fmul_rn(d45.x * code_prescale(4), s);
    dst[5] = __fmul_rn(d45.y * code_prescale(5), s);
    dst[6] = __fmul_rn(d67.x * code_prescale(6), s);
    dst[7] = __fmul_rn(d67.y * code_prescale(7), s);
}

}  // namespace

cudaError_t launch_unpack(int K, int N, const uint32_t *Bq, uint8_t *q, cudaStream_t stream)
{
    const size_t words = (size_t)N * (size_t)(K / 8);
    const unsigned blocks = (unsigned)((words + 255) / 256);
    unpack_kernel<<<blocks, 256, 0, stream>>>(words, Bq, q, kMagicBits);
    return cudaGetLastError();
}

cudaError_t launch_dequant(int K, int N, int gs, const uint32_t *Bq, const float *scales,
                           const float *zeros, float *W, cudaStream_t stream)
{
    const size_t words = (size_t)N * (size_t)(K / 8);
    const unsigned blocks = (unsigned)((words + 255) / 256);
    dequant_kernel<<<blocks, 256, 0, stream>>>(words, K, gs, Bq, scales, zeros, W, kMagicBits);
    return cudaGetLastError();
}

}  // namespace gq4

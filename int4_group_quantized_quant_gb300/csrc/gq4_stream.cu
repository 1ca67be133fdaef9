// gq4_stream.cu -- persistent, bulk-copy (TMA) fed CUDA-core kernels for the
// one-lane (M = 1) decode matvec family: plain, quad routing, RMSNorm
// prologue and SiLU-gated gate/up.
//
// Operation (gerbil moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 and
// WGSL_NORM_MATVEC_INT4): C[n] = sum_k a[k] * (q(n,k) - z) * s.
//
// Decomposition.  At M = 1 the path is one streaming pass over the weights,
// so the kernel is organised around moving bytes:
//   * Persistent grid (about 1-2 CTAs per SM).  CTA b owns one contiguous
//     range of whole columns; ranges are balanced in units of 1, 2 or 4
//     columns so that every copy of scale/zero rows starts 16-byte aligned.
//     Contiguous columns are contiguous bytes in the [N][K/8] layout.
//   * One producer warp streams the range through a ring of S shared-memory
//     slots with cp.async.bulk (global -> shared, completion on an mbarrier).
//     A slot holds `cps` columns of packed codes plus their scale and zero
//     rows (of both matrices for the gated call).
//   * Consumer warps are activation-stationary: lane (w, l) of a column
//     group owns 32-code chunks t = 32w + l (+ 32W r) of K for every column
//     and keeps the 32 matching activations in registers, pre-scaled by
//     16^-p (see gq4_device.cuh).  Shared memory then carries only the
//     weights (0.5 byte per code), read as conflict-free 128-bit loads.
//   * The norm prologue (x = A + A_b, inverse RMS, gain) runs once per CTA
//     while the producer's first copies are in flight.
//   * Per slot a warp handles four weight streams (four columns, or two gate
//     and two up columns), reduces them with an xor reduce-scatter (the same
//     addition tree as a full butterfly for each column), and the W warps of
//     a group combine their partials in warp order through shared memory.
//     Results are deterministic and do not depend on the grid size.
//   * Every mbarrier wait is bounded in time; on expiry the kernel records
//     an error in a device word (gq4_device_error) and leaves.
#include <cstdint>

#include "gq4_device.cuh"
#include "gq4_internal.h"
#include "gq4_tma.cuh"

namespace gq4 {

// Sticky device-side error word (bit 0: a wait for a bulk copy timed out).
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int kStreams = 4;        // weight columns a warp reduces together per slot
constexpr int kMaxR = 2;           // chunks per lane (K <= 32768 on this path)
constexpr int kMaxConsumerWarps = 16;
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;

struct StreamParams {
    int K, N, gs;
    int KC, G;
    int W;            // K-warps per column group
    int Gc;           // column groups
    int cpg;          // columns per group per slot
    int cps;          // columns per slot (Gc * cpg)
    int S;            // ring depth
    int unit;         // column granularity of the balanced split
    int n_units;
    uint32_t slot_bytes;
    uint32_t off_w[2], off_s[2], off_z[2];
    uint32_t off_red, off_norm, off_bar;
    unsigned long long group_magic;
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
    return (int)(((unsigned long long)gc * magic) >> 40);
}

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void record_error(unsigned int bits)
{
    atomicOr(&g_device_error, bits);
}

template <int NMAT, bool NORM, int EPI, int R>
__global__ void __launch_bounds__(kMaxThreads, 1)
stream_matvec_kernel(const __grid_constant__ StreamParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + kMaxStages;
    float *red = reinterpret_cast<float *>(smem + p.off_red);      // [2][Gc][W][4]
    float *red_norm = reinterpret_cast<float *>(smem + p.off_norm); // [Gc][W]

    const int n_consumer_warps = p.Gc * p.W;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- this CTA's column range (whole units) ----
    const int u0 = (int)((long long)p.n_units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)p.n_units * (blockIdx.x + 1) / gridDim.x);
    const int col_begin = u0 * p.unit;
    const int col_end = min(u1 * p.unit, p.N);
    if (col_begin >= col_end) return;  // uniform for the CTA, before any barrier
    const int n_slots_total = (col_end - col_begin + p.cps - 1) / p.cps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], n_consumer_warps);
        }
        mbar_fence_init();
    }
    __syncthreads();

    // =====================================================================
    // Producer warp: stream the column range through the ring.
    // =====================================================================
    if (warp == n_consumer_warps) {
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < n_slots_total; ++i) {
                const int slot = i % p.S;
                if (i >= p.S && !mbar_wait(&empty[slot], ((i / p.S) - 1) & 1)) {
                    record_error(1u);
                    ok = false;
                    break;
                }
                const int c0 = col_begin + i * p.cps;
                const int nc = min(p.cps, col_end - c0);
                const uint32_t w_bytes = (uint32_t)nc * (uint32_t)p.KC * 16u;
                const uint32_t s_bytes = ((uint32_t)nc * (uint32_t)p.G * 4u) & ~15u;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)NMAT * (w_bytes + 2u * s_bytes));
                unsigned char *dst = smem + (size_t)slot * p.slot_bytes;
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    bulk_g2s(dst + p.off_w[m], p.Bq[m] + (size_t)c0 * p.KC, w_bytes, &full[slot]);
                    if (s_bytes) {
                        bulk_g2s(dst + p.off_s[m], p.scales[m] + (size_t)c0 * p.G, s_bytes, &full[slot]);
                        bulk_g2s(dst + p.off_z[m], p.zeros[m] + (size_t)c0 * p.G, s_bytes, &full[slot]);
                    }
                }
                issued = i + 1;
            }
            if (!ok) {
                // leave no copy in flight into this CTA's shared memory
                for (int i = (issued > p.S ? issued - p.S : 0); i < issued; ++i)
                    (void)mbar_wait(&full[i % p.S], (i / p.S) & 1);
            }
        }
        return;
    }

    // =====================================================================
    // Consumer warps.
    // =====================================================================
    const int g = warp / p.W;     // column group
    const int w = warp - g * p.W; // K-warp within the group
    const int bar_id = 1 + g;
    const int group_threads = p.W * 32;

    int t[R];
    bool has[R];
    int grp[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        t[r] = w * 32 + lane + r * p.W * 32;
        has[r] = t[r] < p.KC;
        grp[r] = has[r] ? chunk_group(t[r], p.group_magic) : 0;
    }

    // ---- activations of the owned chunks, in registers ----
    f32x2 act[R][16];
    float sumsq = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (has[r]) {
                const size_t k = (size_t)t[r] * 32 + (size_t)j * 4;
                v = *reinterpret_cast<const float4 *>(p.A + k);
                if constexpr (NORM) {
                    if (p.A_b) {
                        const float4 b = *reinterpret_cast<const float4 *>(p.A_b + k);
                        v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
                    }
                    sumsq = fmaf(v.x, v.x, sumsq);
                    sumsq = fmaf(v.y, v.y, sumsq);
                    sumsq = fmaf(v.z, v.z, sumsq);
                    sumsq = fmaf(v.w, v.w, sumsq);
                }
            }
            act[r][2 * j] = pack2(v.x, v.y);
            act[r][2 * j + 1] = pack2(v.z, v.w);
        }
    }

    if constexpr (NORM) {
        // inverse RMS over all K: warp butterfly, then warps in order
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, off);
        if (p.W > 1) {
            if (lane == 0) red_norm[g * p.W + w] = sumsq;
            named_barrier(bar_id, group_threads);
            sumsq = 0.0f;
            for (int i = 0; i < p.W; ++i) sumsq += red_norm[g * p.W + i];
        }
        const float inv = 1.0f / sqrtf(sumsq / (float)p.K + p.eps);
        const bool write_side = blockIdx.x == 0 && g == 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (!has[r]) continue;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const size_t k = (size_t)t[r] * 32 + (size_t)j * 4;
                const float2 lo = unpack2(act[r][2 * j]);
                const float2 hi = unpack2(act[r][2 * j + 1]);
                float4 x = make_float4(lo.x, lo.y, hi.x, hi.y);
                if (write_side && p.residual_out) *reinterpret_cast<float4 *>(p.residual_out + k) = x;
                const float4 gn = *reinterpret_cast<const float4 *>(p.W_norm + k);
                x.x = (x.x * inv) * gn.x; x.y = (x.y * inv) * gn.y;
                x.z = (x.z * inv) * gn.z; x.w = (x.w * inv) * gn.w;
                if (write_side && p.norm_out) *reinterpret_cast<float4 *>(p.norm_out + k) = x;
                act[r][2 * j] = pack2(x.x, x.y);
                act[r][2 * j + 1] = pack2(x.z, x.w);
            }
        }
    }
    // pre-scale by 16^-p (exact): both halves of a word sit at p = 0, 1, 2, 3
    {
        const f32x2 ps01 = pack2(code_prescale(0), code_prescale(1));
        const f32x2 ps23 = pack2(code_prescale(2), code_prescale(3));
        const f32x2 zero2 = pack2(0.0f, 0.0f);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < 16; ++j) act[r][j] = fma2(act[r][j], (j & 1) ? ps23 : ps01, zero2);
    }

    const f32x2 nmagic2 = neg_magic2();
    // A consumer whose bounded wait expires keeps walking the slots (releasing
    // them and joining its group's barriers, so no sibling warp is left
    // waiting) but stops waiting and reading; its outputs become NaN.
    bool failed = false;

    for (int i = 0; i < n_slots_total; ++i) {
        const int slot = i % p.S;
        const int c0 = col_begin + i * p.cps;
        const int nc = min(p.cps, col_end - c0);
        if (!failed && !mbar_wait(&full[slot], (i / p.S) & 1)) {
            record_error(1u);
            failed = true;
        }
        const unsigned char *sl = smem + (size_t)slot * p.slot_bytes;
        const int s_smem_floats = (int)((((uint32_t)nc * (uint32_t)p.G * 4u) & ~15u) >> 2);

        float part[kStreams];
#pragma unroll
        for (int q = 0; q < kStreams; ++q) {
            const int mat = NMAT == 2 ? (q >> 1) : 0;
            const int lc = NMAT == 2 ? g * 2 + (q & 1) : g * 4 + q;  // column within the slot
            float acc = 0.0f;
            if (lc < nc && !failed) {
                const uint4 *wsm = reinterpret_cast<const uint4 *>(sl + p.off_w[mat]);
                const float *ssm = reinterpret_cast<const float *>(sl + p.off_s[mat]);
                const float *zsm = reinterpret_cast<const float *>(sl + p.off_z[mat]);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (!has[r]) continue;
                    const uint4 wq = wsm[(size_t)lc * p.KC + t[r]];
                    const int si = lc * p.G + grp[r];
                    float sc, zr;
                    if (si < s_smem_floats) {
                        sc = ssm[si];
                        zr = zsm[si];
                    } else {  // the last few floats of the arrays when N*G is not a multiple of 4
                        sc = __ldg(p.scales[mat] + (size_t)c0 * p.G + si);
                        zr = __ldg(p.zeros[mat] + (size_t)c0 * p.G + si);
                    }
                    const ZeroPairs zp = scaled_zero(zr);
                    f32x2 inner = pack2(0.0f, 0.0f);
#pragma unroll
                    for (int wd = 0; wd < 4; ++wd) {
                        const uint32_t word = wd == 0 ? wq.x : wd == 1 ? wq.y : wd == 2 ? wq.z : wq.w;
                        const DiffPairs d = code_minus_zero(word, zp, nmagic2);
                        inner = fma2(act[r][4 * wd + 0], d.d01, inner);
                        inner = fma2(act[r][4 * wd + 1], d.d23, inner);
                        inner = fma2(act[r][4 * wd + 2], d.d45, inner);
                        inner = fma2(act[r][4 * wd + 3], d.d67, inner);
                    }
                    const float2 v = unpack2(inner);
                    acc = fmaf(sc, v.x + v.y, acc);
                }
            }
            part[q] = acc;
        }
        // the slot's shared memory has been read: release it to the producer
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);

        // ---- reduce-scatter of the four streams across the warp ----
        // step 16: lanes < 16 keep streams 0,1; lanes >= 16 keep streams 2,3
        const bool hi16 = (lane & 16) != 0;
        float k0 = hi16 ? part[2] : part[0];
        float k1 = hi16 ? part[3] : part[1];
        const float s0 = hi16 ? part[0] : part[2];
        const float s1 = hi16 ? part[1] : part[3];
        k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
        k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
        // step 8: lanes with bit 3 clear keep the first, others the second
        const bool hi8 = (lane & 8) != 0;
        float v = hi8 ? k1 : k0;
        v += __shfl_xor_sync(0xffffffffu, hi8 ? k0 : k1, 8);
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        // lane 0 -> stream 0, lane 8 -> stream 1, lane 16 -> stream 2, lane 24 -> stream 3
        const int q_of_lane = ((lane >> 4) << 1) | ((lane >> 3) & 1);

        float total = v;
        if (p.W > 1) {
            float *rb = red + ((size_t)(i & 1) * p.Gc + g) * p.W * kStreams;
            if ((lane & 7) == 0) rb[w * kStreams + q_of_lane] = v;
            named_barrier(bar_id, group_threads);
            if (w != 0) continue;
            if ((lane & 7) == 0) {
                total = 0.0f;
                for (int k = 0; k < p.W; ++k) total += rb[k * kStreams + q_of_lane];
            }
        }

        if (failed) total = __int_as_float(0x7fffffff);

        // ---- epilogue: lanes 0, 8, 16, 24 of warp 0 of the group ----
        if constexpr (EPI == kEpiGated) {
            const float u = __shfl_down_sync(0xffffffffu, total, 16);  // up partner
            if ((lane & 7) == 0 && lane < 16) {
                const int lc = g * 2 + (lane >> 3);
                if (lc < nc) {
                    const float gv = total;
                    p.out[0][c0 + lc] = gv / (1.0f + expf(-gv)) * u;
                }
            }
        } else {
            if ((lane & 7) == 0) {
                const int lc = g * 4 + q_of_lane;
                if (lc < nc) {
                    const int col = c0 + lc;
                    if constexpr (EPI == kEpiQuad) {
                        const int seg = col < p.seg_start[1] ? 0 : col < p.seg_start[2] ? 1
                                      : col < p.seg_start[3] ? 2 : 3;
                        p.out[seg][col - p.seg_start[seg]] = total;
                    } else {
                        p.out[0][col] = total;
                    }
                }
            }
        }
    }
}

int gcd_int(int a, int b)
{
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

uint32_t round_up(uint32_t x, uint32_t a)
{
    return (x + a - 1) / a * a;
}

template <int NMAT, bool NORM, int EPI, int R>
cudaError_t launch_stream_variant(const StreamParams &prm, int threads, size_t smem,
                                  cudaStream_t stream)
{
    auto kern = stream_matvec_kernel<NMAT, NORM, EPI, R>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    int dev = 0, sms = 0, per_sm = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem)) !=
        cudaSuccess)
        return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int grid = sms * (per_sm > 2 ? 2 : per_sm);
    if (grid > prm.n_units) grid = prm.n_units;
    kern<<<grid, threads, smem, stream>>>(prm);
    return cudaGetLastError();
}

template <int NMAT, bool NORM, int EPI>
cudaError_t launch_stream_r(const StreamParams &prm, int R, int threads, size_t smem,
                            cudaStream_t stream)
{
    return R == 1 ? launch_stream_variant<NMAT, NORM, EPI, 1>(prm, threads, smem, stream)
                  : launch_stream_variant<NMAT, NORM, EPI, 2>(prm, threads, smem, stream);
}

}  // namespace

bool stream_path_supported(const Call &call)
{
    if (call.M != 1) return false;
    const int KC = call.K / 32;
    if (KC > kMaxR * kMaxConsumerWarps * 32) return false;
    for (int m = 0; m < call.nmat; ++m) {
        if ((reinterpret_cast<uintptr_t>(call.scales[m]) & 15u) != 0) return false;
        if ((reinterpret_cast<uintptr_t>(call.zeros[m]) & 15u) != 0) return false;
    }
    return true;
}

cudaError_t launch_stream(const Call &call, cudaStream_t stream)
{
    StreamParams prm{};
    prm.K = call.K;
    prm.N = call.N;
    prm.gs = call.gs;
    prm.KC = call.K / 32;
    prm.G = call.K / call.gs;
    const unsigned long long cpgrp = (unsigned long long)(call.gs / 32);
    prm.group_magic = ((1ull << 40) + cpgrp - 1) / cpgrp;

    int R = (prm.KC + 32 * kMaxConsumerWarps - 1) / (32 * kMaxConsumerWarps);
    if (R < 1) R = 1;
    prm.W = (prm.KC + 32 * R - 1) / (32 * R);
    prm.Gc = prm.W >= 8 ? 1 : 8 / prm.W;
    prm.cpg = call.nmat == 2 ? 2 : 4;
    prm.cps = prm.Gc * prm.cpg;
    prm.unit = 4 / gcd_int(prm.G, 4);
    if (prm.cps % prm.unit != 0) return cudaErrorInvalidValue;  // not reached for cpg >= 2 and unit <= 2
    prm.n_units = (call.N + prm.unit - 1) / prm.unit;

    // slot layout
    uint32_t off = 0;
    const uint32_t sz_bytes = round_up((uint32_t)prm.cps * prm.G * 4u, 16u);
    for (int m = 0; m < call.nmat; ++m) {
        prm.off_w[m] = off;
        off += (uint32_t)prm.cps * prm.KC * 16u;
        prm.off_s[m] = off;
        off += sz_bytes;
        prm.off_z[m] = off;
        off += sz_bytes;
    }
    prm.slot_bytes = round_up(off, 128u);
    const uint32_t budget = (prm.Gc * prm.W <= 8) ? 96u * 1024u : 192u * 1024u;
    int S = (int)(budget / prm.slot_bytes);
    if (S > kMaxStages) S = kMaxStages;
    if (S < 2) S = 2;
    prm.S = S;
    prm.off_red = round_up((uint32_t)S * prm.slot_bytes, 128u);
    prm.off_norm = prm.off_red + round_up(2u * prm.Gc * prm.W * kStreams * 4u, 16u);
    prm.off_bar = prm.off_norm + round_up((uint32_t)prm.Gc * prm.W * 4u, 16u);
    const size_t smem = prm.off_bar + 2 * kMaxStages * sizeof(uint64_t);
    if (smem > 227u * 1024u) return cudaErrorInvalidValue;

    prm.A = call.A;
    if (call.norm) {
        prm.A_b = call.norm->A_b;
        prm.W_norm = call.norm->W_norm;
        prm.eps = call.norm->eps;
        prm.residual_out = call.norm->residual_out;
        prm.norm_out = call.norm->norm_out;
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
    const int threads = (prm.Gc * prm.W + 1) * 32;
    const bool norm = call.norm != nullptr;
    switch (call.epi) {
    case kEpiStore:
        return norm ? launch_stream_r<1, true, kEpiStore>(prm, R, threads, smem, stream)
                    : launch_stream_r<1, false, kEpiStore>(prm, R, threads, smem, stream);
    case kEpiQuad:
        return launch_stream_r<1, false, kEpiQuad>(prm, R, threads, smem, stream);
    case kEpiGated:
        return norm ? launch_stream_r<2, true, kEpiGated>(prm, R, threads, smem, stream)
                    : launch_stream_r<2, false, kEpiGated>(prm, R, threads, smem, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t read_device_error(unsigned int *bits, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(bits, g_device_error, sizeof(unsigned int));
    if (err != cudaSuccess || !clear) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

}  // namespace gq4

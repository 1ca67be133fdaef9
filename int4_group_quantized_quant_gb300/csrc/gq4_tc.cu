// gq4_tc.cu -- the batched-lane (16 <= M <= 32) int4 group-quantized matvec
// family on the 5th-generation tensor core: plain, quad routing, RMSNorm
// prologue and SiLU-gated gate/up.
//
// Operation (gerbil moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 and
// WGSL_NORM_MATVEC_INT4, batched over decode lanes): C[m][n] = sum_k
// a[m][k] * (q(n,k) - z) * s.  With M lanes sharing every weight the product
// is a small GEMM, D[n][m] = W[n][:] . A[m][:], computed here in bf16 with f32
// accumulation: the weights are dequantized in registers to bf16 and the MMA
// runs with the weight tile as the M=128 operand and the lanes as N (16/32).
//
// Decomposition.
//   * Tiles of TR <= 128 weight columns (one MMA row per column).  A thread-
//     block cluster of KS CTAs owns a tile; its CTAs split K in whole 256-code
//     stages, and their f32 partial tiles are summed through distributed
//     shared memory in rank order (deterministic, no global scratch).
//   * Producer warp: lane 0 issues a 2-D tensor-map copy of the tile's packed
//     codes for a stage (TR rows x 128 bytes, 128-byte swizzle, zero fill
//     past K and N) as soon as a ring slot is free; the 32 lanes copy the
//     stage's raw scales and zeros with 4-byte cp.async (zero fill past N and
//     K), whose completion arrives on the same barrier as the tensor copy.
//     (Scale rows of K/gs floats need not be 16-byte multiples, so they are
//     not described by a tensor map.)
//   * Dequant warps (8): two per TMEM lane quarter.  A thread owns one row
//     and half of each 64-code K-block; when its scale group changes it turns
//     (s, z) into bf16 pairs (128 + zi, s, (zi - z) * s) with zi =
//     round(clamp(z, 0, 15)).  Per word, four LOP3 magic extractions
//     give bf16 pairs (128+q), an exact bf16 subtraction gives q - zi, and an
//     fma gives (q - zi)*s + (zi - z)*s = (q - z)*s rounded once to bf16.  The
//     16 results go straight to tensor memory (tcgen05.st): the dequantized
//     tile never touches shared memory.
//   * One MMA thread: per K-block, four tcgen05.mma (kind::f16, 128 x N x 16)
//     per matrix, A from tensor memory, B (the lanes' activations) from
//     shared memory, D accumulating in tensor memory; tcgen05.commit frees
//     the K-block's tensor-memory slot and, per tile, hands the accumulator
//     to the epilogue.
//   * Epilogue warps (4): tcgen05.ld of the accumulator, the split-K sum
//     across the cluster, then the store / quad routing / silu(g)*u.
//   * Activations (and the RMSNorm prologue) for the CTA's K range are
//     staged once, in bf16, in the canonical K-major 128-byte swizzled layout
//     the MMA reads.  The codes of a word are stored in the order
//     (0,4,1,5,2,6,3,7) -- the order the magic extraction yields -- and the
//     activations are permuted the same way, so the dot product is unchanged.
//   * Every wait is bounded; on expiry the kernel records an error in a
//     device word (gq4_device_error), stops waiting and leaves.
#include <cuda.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "gq4_host.h"
#include "gq4_internal.h"
#include "gq4_tcgen05.cuh"

namespace gq4 {

// Sticky device-side error word of this path (bit 1: a wait timed out).
__device__ unsigned int g_tc_error = 0;

namespace {

constexpr int kDqWarps = 8;     // warps 0..7
constexpr int kEpWarps = 4;     // warps 8..11
constexpr int kPrWarp = 12;     // warp 12
constexpr int kMmaWarp = 13;    // warp 13
constexpr int kThreads = 14 * 32;
constexpr int kEpBase = kDqWarps * 32;
constexpr int kMaxNW = 12;      // tensor-memory slots of dequantized K-blocks (most)
constexpr int kMaxKs = 8;       // CTAs per cluster (split-K ranks), most
constexpr int kStageK = 256;    // codes per stage along K
constexpr int kBlockK = 64;     // codes per K-block (one 128-byte bf16 row)
constexpr int kMaxStages = 16;
constexpr int kMaxGps = 8;      // scale groups a stage can touch (gs >= 32)
constexpr uint32_t kMinSmem = 120u * 1024u;  // forces one CTA per SM (tensor memory)

struct TcParams {
    CUtensorMap codes[2];          // [N][K/8] u32, box {32, TR}, 128-byte swizzle
    CUtensorMap sz[2][2];          // scales / zeros [mat][s|z] as super-rows of P rows:
                                   // [Q][P*G] f32, box {BW, TR/P}
    int M, K, N, gs, G;
    int TR;                        // rows per tile
    int n_tiles, n_clusters, ks;
    int n_st;                      // stages over K
    int S;                         // ring depth
    int gps;                       // most groups a stage touches
    int P, Q, BW;                  // rows per super-row, whole super-rows, box width (groups)
    int logP;                      // log2(P)
    unsigned long long gmagic;     // ceil(2^40 / (gs/32)): chunk index -> group, exactly
    uint32_t off_act, off_ring, stage_bytes, codes_bytes;
    uint32_t sz_box_bytes, sz_box_stride, off_sz, off_tail;
    uint32_t off_red, off_misc, off_bar;
    uint32_t magic_bf16;           // 0x43004300, read from the parameter bank
    const float *A;
    const float *A_b;
    const float *W_norm;
    float eps;
    float *residual_out;
    float *norm_out;
    const float *scales[2];
    const float *zeros[2];
    float *out[4];
    int seg_start[4];
    int seg_len[4];
};

struct Shared {
    uint64_t *full, *empty, *w_full, *w_empty, *acc_full, *acc_empty;
    uint64_t *act_ready, *red_full, *red_empty, *norm_full, *drain;
    float *part;      // [32] this CTA's norm partial sums
    uint32_t *tmem;   // allocated tensor-memory base
    int *abort;
};

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_cluster()
{
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// Non-blocking test of an mbarrier phase (no suspension).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait on an mbarrier phase.  Gives up (false) when another thread of
// the CTA has already given up, or after the time limit (then it records the
// error and tells the CTA).  `cluster` waits acquire at cluster scope; CTA
// waits poll with test_wait rather than suspend in try_wait, whose wake-up
// after the phase completes cost ~0.3 us per wait here.
__device__ __noinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort, bool cluster)
{
    auto ready = [&]() { return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_test(bar, parity); };
    if (ready()) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (ready()) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(&g_tc_error, 2u);
            return false;
        }
    }
}

// The MMA thread's wait on a K-block slot: a bounded poll with test_wait
// (no suspension); the same change made the GEMM kernel ~9% faster.
__device__ __forceinline__ bool tc_poll(uint64_t *bar, uint32_t parity, volatile int *abort)
{
    const unsigned long long t0 = global_timer_ns();
    for (unsigned int i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 255u) == 255u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(&g_tc_error, 2u);
                return false;
            }
        }
    }
}

// Wait without giving up early on another thread's abort (used to drain
// copies and MMAs in flight before the CTA leaves); still bounded.
__device__ __forceinline__ void tc_drain_wait(uint64_t *bar, uint32_t parity)
{
    (void)mbar_wait(bar, parity);
}

// Scale group of 32-code chunk c (c < 2^19): c / (gs/32) by multiply-shift.
__device__ __forceinline__ int chunk_group(int c, unsigned long long gmagic)
{
    return (int)(((unsigned long long)c * gmagic) >> 40);
}

// Output epilogue for one (lane, column).
template <int EPI>
__device__ __forceinline__ void store_out(const TcParams &p, int m, int col, float v0, float v1)
{
    if constexpr (EPI == kEpiGated) {
        p.out[0][(size_t)m * p.N + col] = v0 / (1.0f + expf(-v0)) * v1;
    } else if constexpr (EPI == kEpiQuad) {
        const int seg = col < p.seg_start[1] ? 0 : col < p.seg_start[2] ? 1 : col < p.seg_start[3] ? 2 : 3;
        p.out[seg][(size_t)m * p.seg_len[seg] + (col - p.seg_start[seg])] = v0;
    } else {
        p.out[0][(size_t)m * p.N + col] = v0;
    }
}

// Eight activations a[0..7] of one 8-code chunk as bf16 in the word's code
// order (0,4,1,5,2,6,3,7).
__device__ __forceinline__ uint4 pack_chunk(const float4 &lo, const float4 &hi)
{
    uint4 r;
    r.x = bf16x2_pack(lo.x, hi.x);
    r.y = bf16x2_pack(lo.y, hi.y);
    r.z = bf16x2_pack(lo.z, hi.z);
    r.w = bf16x2_pack(lo.w, hi.w);
    return r;
}

// Byte offset of chunk c (0..7) of lane row m in one K-block of the
// activation operand (MP rows of 128 bytes, 8-row atoms of 1024 bytes).
__device__ __forceinline__ uint32_t act_chunk_offset(int m, int c)
{
    return (uint32_t)((m >> 3) * 1024 + (m & 7) * 128 + ((c ^ (m & 7)) << 4));
}

template <int MP, int NMAT, bool NORM, int EPI>
__global__ void __launch_bounds__(kThreads, 1) tc_matvec_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base (128-byte swizzle atoms)
    const uint32_t raw_s = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);

    Shared sh;
    {
        uint64_t *b = reinterpret_cast<uint64_t *>(smem + p.off_bar);
        sh.full = b;
        sh.empty = b + kMaxStages;
        sh.w_full = b + 2 * kMaxStages;
        sh.w_empty = sh.w_full + kMaxNW;
        sh.acc_full = sh.w_empty + kMaxNW;
        sh.acc_empty = sh.acc_full + 2;
        sh.act_ready = sh.acc_empty + 2;
        sh.red_full = sh.act_ready + 1;
        sh.red_empty = sh.red_full + 1;
        sh.norm_full = sh.red_empty + 1;
        sh.drain = sh.norm_full + 1;
        sh.part = reinterpret_cast<float *>(smem + p.off_misc);
        sh.tmem = reinterpret_cast<uint32_t *>(smem + p.off_misc + 128);
        sh.abort = reinterpret_cast<int *>(smem + p.off_misc + 132);
    }
    volatile int *abort = sh.abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ks = p.ks;
    const int rank = ks > 1 ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / ks;
    // this rank's stages along K
    const int st0 = (int)((long long)p.n_st * rank / ks);
    const int st1 = (int)((long long)p.n_st * (rank + 1) / ks);
    const int spr = st1 - st0;
    const int KBr = spr * (kStageK / kBlockK);
    // this cluster's tiles: cid, cid + n_clusters, ...
    const int n_tl = cid < p.n_tiles ? (p.n_tiles - cid + p.n_clusters - 1) / p.n_clusters : 0;
    const int n_stages_total = n_tl * spr;
    // tensor memory: kNW dequantized K-blocks per matrix, two accumulators per matrix
    constexpr int kNW = NMAT == 1 ? 12 : 6;
    // K-blocks per hand-off step between the dequant warps and the MMA thread
    // (one wait, one arrival and one commit per step, not per K-block: each
    // barrier round trip costs ~0.2 us, more than a K-block's MMAs), and the
    // steps tensor memory holds
    constexpr int kKPS = NMAT == 1 ? 4 : 2;
    constexpr int kNS = kNW / kKPS;
    static_assert(kNW % kKPS == 0 && kNS <= kMaxNW, "tensor-memory steps");
    constexpr uint32_t kTmemCols = 512u;
    static_assert(NMAT * kNW * 32 + NMAT * 2 * 32 <= (int)kTmemCols, "tensor-memory map");

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.S; ++s) {
            mbar_init(&sh.full[s], 32);  // the producer lanes' cp.async arrivals
            mbar_init(&sh.empty[s], kDqWarps);
        }
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&sh.w_full[s], kDqWarps);
            mbar_init(&sh.w_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.acc_full[b], 1);
            mbar_init(&sh.acc_empty[b], kEpWarps);
        }
        mbar_init(sh.act_ready, kDqWarps);
        mbar_init(sh.red_full, ks);
        mbar_init(sh.red_empty, ks);
        mbar_init(sh.norm_full, ks);
        mbar_init(sh.drain, 1);
        *sh.abort = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(sh.tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *sh.tmem;
    // Cluster barrier in two halves: every thread arrives now; a thread waits
    // (peers' barriers initialised) only before its first access to a peer,
    // so the copies start at once.
    if (ks > 1) cluster_arrive();
    bool cwaited = false;

    // tensor-memory columns: W slots, then two accumulators per matrix
    auto w_col = [&](int mat, int slot) { return (uint32_t)((mat * kNW + slot) * 32); };
    auto acc_col = [&](int mat, int b) { return (uint32_t)(NMAT * kNW * 32 + (mat * 2 + b) * 32); };

    // =====================================================================
    // Producer warp: codes, scales and zeros (tensor-map copies; cp.async
    // for the at most P-1 rows past the last whole super-row).
    // =====================================================================
    if (warp == kPrWarp) {
        if (lane == 0) {
#pragma unroll
            for (int mat = 0; mat < NMAT; ++mat) {
                prefetch_tensormap(&p.codes[mat]);
                prefetch_tensormap(&p.sz[mat][0]);
                prefetch_tensormap(&p.sz[mat][1]);
            }
        }
        bool ok = true;
        int issued = 0;
        // ring position and (tile, stage-in-rank) of stage i, kept incrementally
        int slot = 0, phase = 0, tl = 0, sir = 0;
        for (int i = 0; i < n_stages_total; ++i) {
            if (i >= p.S) {
                bool got = true;
                if (lane == 0) got = tc_wait(&sh.empty[slot], phase ^ 1, abort, false);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    ok = false;
                    break;
                }
            }
            unsigned char *stage = smem + p.off_ring + (size_t)slot * p.stage_bytes;
            const int k0 = (st0 + sir) * kStageK;
            const int row0 = (cid + tl * p.n_clusters) * p.TR;
            const int g0 = chunk_group(k0 >> 5, p.gmagic);
            if (lane == 0) {
                mbar_expect_tx(&sh.full[slot], (uint32_t)NMAT * (p.codes_bytes + 2u * p.P * p.sz_box_bytes));
#pragma unroll
                for (int mat = 0; mat < NMAT; ++mat) {
                    tma_load_2d(stage + mat * p.codes_bytes, &p.codes[mat], k0 / 8, row0, &sh.full[slot]);
#pragma unroll
                    for (int arr = 0; arr < 2; ++arr)
                        for (int rho = 0; rho < p.P; ++rho) {
                            const int x = (rho * p.G + g0) & ~3;
                            tma_load_2d(stage + p.off_sz + ((mat * 2 + arr) * p.P + rho) * p.sz_box_stride,
                                        &p.sz[mat][arr], x, row0 >> p.logP, &sh.full[slot]);
                        }
                }
            }
            // rows past the last whole super-row (only in the last tile)
            const int tail0 = p.P * p.Q;
            if (tail0 < p.N && row0 + p.TR > tail0) {
                const int n_tail = p.N - tail0;  // < P
                const int g_last = chunk_group((min(k0 + kStageK, p.K) - 1) >> 5, p.gmagic);
                const int per = n_tail * p.gps;
                for (int it = lane; it < NMAT * 2 * per; it += 32) {
                    const int ma = it / per;            // mat * 2 + arr
                    const int rem = it - ma * per;
                    const int t = rem / p.gps;
                    const int gl = rem - t * p.gps;
                    const int off = (t * p.G + g0) & 3;
                    const bool valid = k0 < p.K && g0 + gl <= g_last;
                    const float *src = (ma & 1) ? p.zeros[ma >> 1] : p.scales[ma >> 1];
                    float *d = reinterpret_cast<float *>(stage + p.off_tail) + (ma * 4 + t) * p.BW + off + gl;
                    cp_async_4(d, src + (valid ? (size_t)(tail0 + t) * p.G + g0 + gl : 0), valid);
                }
            }
            cp_async_mbar_arrive(&sh.full[slot]);
            issued = i + 1;
            if (++slot == p.S) {
                slot = 0;
                phase ^= 1;
            }
            if (++sir == spr) {
                sir = 0;
                ++tl;
            }
        }
        if (!ok && lane == 0) {
            // leave no copy in flight into this CTA's shared memory
            for (int i = (issued > p.S ? issued - p.S : 0); i < issued; ++i)
                tc_drain_wait(&sh.full[i % p.S], (i / p.S) & 1);
        }
    }

    // =====================================================================
    // Dequant warps: activation staging first, then K-blocks into TMEM.
    // =====================================================================
    else if (warp < kDqWarps) {
        const int tid = threadIdx.x;
        const int k_base = st0 * kStageK;
        const int n_chunks = KBr * 8;                 // 8-code chunks of this rank's K range
        constexpr int TPL = (kDqWarps * 32) / MP;     // threads per lane row
        const int m = tid / TPL;
        const int sub = tid % TPL;
        unsigned char *act = smem + p.off_act;
        // the norm's side outputs are written once, spread over the clusters:
        // chunk c of lane m by cluster (m * n_chunks + c) mod n_clusters
        auto writer = [&](int mm, int c) { return (mm * n_chunks + c) % p.n_clusters == cid; };
        bool ok = true;
        // the activations may be the previous kernel's outputs
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if constexpr (NORM) {
            // One pass over A, A_b and W_norm: x = A + A_b (x itself to
            // residual_out), its square sum, and bf16(x * W_norm) staged as
            // the operand.  The inverse RMS is a per-lane scalar: the
            // epilogue applies it to each finished dot product, once the
            // cluster's square sums are in, and writes norm_out (exact f32,
            // from x recomputed) meanwhile.  Staging thus needs no cluster
            // round trip.
            constexpr int kU = 4;
            const size_t row_off = (size_t)(m < p.M ? m : 0) * p.K;
            const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            float part = 0.0f;
            for (int c0 = sub; c0 < n_chunks; c0 += kU * TPL) {
                float4 x[kU][2], b[kU][2], g[kU][2];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + u * TPL;
                    const int k = k_base + 8 * c;
                    const bool in = c < n_chunks && m < p.M && k < p.K;
                    const float4 *a4 = reinterpret_cast<const float4 *>(p.A + row_off + (in ? k : 0));
                    const float4 *b4 = reinterpret_cast<const float4 *>(
                        (p.A_b ? p.A_b : p.A) + row_off + (in ? k : 0));
                    const float4 *w4 = reinterpret_cast<const float4 *>(p.W_norm + (in ? k : 0));
                    x[u][0] = in ? __ldg(a4) : z4;
                    x[u][1] = in ? __ldg(a4 + 1) : z4;
                    b[u][0] = in && p.A_b ? __ldg(b4) : z4;
                    b[u][1] = in && p.A_b ? __ldg(b4 + 1) : z4;
                    g[u][0] = in ? __ldg(w4) : z4;
                    g[u][1] = in ? __ldg(w4 + 1) : z4;
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + u * TPL;
                    if (c >= n_chunks) continue;
                    const int k = k_base + 8 * c;
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        x[u][v].x += b[u][v].x; x[u][v].y += b[u][v].y;
                        x[u][v].z += b[u][v].z; x[u][v].w += b[u][v].w;
                    }
                    if (p.residual_out && m < p.M && k < p.K && writer(m, c)) {
                        float4 *ro = reinterpret_cast<float4 *>(p.residual_out + row_off + k);
                        ro[0] = x[u][0];
                        ro[1] = x[u][1];
                    }
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        part = fmaf(x[u][v].x, x[u][v].x, part);
                        part = fmaf(x[u][v].y, x[u][v].y, part);
                        part = fmaf(x[u][v].z, x[u][v].z, part);
                        part = fmaf(x[u][v].w, x[u][v].w, part);
                        x[u][v].x *= g[u][v].x; x[u][v].y *= g[u][v].y;
                        x[u][v].z *= g[u][v].z; x[u][v].w *= g[u][v].w;
                    }
                    *reinterpret_cast<uint4 *>(act + (size_t)(c >> 3) * (MP * 128) + act_chunk_offset(m, c & 7)) =
                        pack_chunk(x[u][0], x[u][1]);
                }
            }
            // fixed-order sum over the TPL threads of the row (consecutive lanes)
#pragma unroll
            for (int off = TPL / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            if (sub == 0) sh.part[m] = part;
            named_barrier(1, kDqWarps * 32);
            if (ks > 1) cluster_wait();  // peers' barriers are initialised
            cwaited = true;
            if (tid == 0) {
                // this CTA's square sums, released to every rank's epilogue
                fence_acq_rel_cluster();
                for (int j = 0; j < ks; ++j) mbar_arrive_cluster(dsmem_addr(smem_addr(sh.norm_full), j));
            }
        } else {
            // batches of kU chunks: all loads issued before the first conversion
            constexpr int kU = 4;
            const float4 *arow = reinterpret_cast<const float4 *>(p.A + (size_t)(m < p.M ? m : 0) * p.K);
            for (int c0 = sub; c0 < n_chunks; c0 += kU * TPL) {
                float4 x[kU][2];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + u * TPL;
                    const int k = k_base + 8 * c;
                    if (c < n_chunks && m < p.M && k < p.K) {
                        x[u][0] = __ldg(arow + k / 4);
                        x[u][1] = __ldg(arow + k / 4 + 1);
                    } else {
                        x[u][0] = x[u][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + u * TPL;
                    if (c < n_chunks)
                        *reinterpret_cast<uint4 *>(act + (size_t)(c >> 3) * (MP * 128) + act_chunk_offset(m, c & 7)) =
                            pack_chunk(x[u][0], x[u][1]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sh.act_ready);

        // ---- K-blocks ----
        const int q4 = warp & 3;
        const int h = warp >> 2;
        const int r = 32 * q4 + lane;
        const bool warp_live = 32 * q4 < p.TR;   // warp-uniform
        const bool row_in_tile = r < p.TR;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const uint32_t magic = p.magic_bf16;
        int kbg = 0;  // K-blocks so far (tensor-memory slot sequence)
        const int rho = r & (p.P - 1);
        const int srow = r >> p.logP;
        int slot = 0, phase = 0, tl = 0, sir = 0;
        for (int i = 0; ok && i < n_stages_total; ++i) {
            // The last stage lets the next kernel in the stream be scheduled
            // (once every CTA has done so or left); earlier, a third kernel
            // could queue for SMs ahead of the second.
            if (i == n_stages_total - 1 && threadIdx.x == 0)
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            // warp-uniform outcome: the collective tensor-memory stores below
            // need every lane
            if (!__all_sync(0xffffffffu, tc_wait(&sh.full[slot], phase, abort, false))) {
                ok = false;
                break;
            }
            const int k0 = (st0 + sir) * kStageK;
            const int c0 = k0 >> 5;  // first 32-code chunk of the stage
            const int g0 = chunk_group(c0, p.gmagic);
            const unsigned char *stage = smem + p.off_ring + (size_t)slot * p.stage_bytes;
            // this row's scales and zeros in the stage: box of residue r % P,
            // super-row r / P (or the tail area), columns from `off`
            const int g_last = chunk_group((min(k0 + kStageK, p.K) - 1) >> 5, p.gmagic);
            const int R = (cid + tl * p.n_clusters) * p.TR + r;
            const bool row_valid = row_in_tile && R < p.N && k0 < p.K;
            const int off = (rho * p.G + g0) & 3;
            const float *s_src[NMAT], *z_src[NMAT];
#pragma unroll
            for (int mat = 0; mat < NMAT; ++mat) {
                if (R >= p.P * p.Q) {
                    const int t = R - p.P * p.Q;
                    const float *tail = reinterpret_cast<const float *>(stage + p.off_tail);
                    s_src[mat] = tail + ((mat * 2 + 0) * 4 + t) * p.BW + off;
                    z_src[mat] = tail + ((mat * 2 + 1) * 4 + t) * p.BW + off;
                } else {
                    const float *box0 = reinterpret_cast<const float *>(
                        stage + p.off_sz + ((mat * 2 + 0) * p.P + rho) * p.sz_box_stride);
                    const float *box1 = reinterpret_cast<const float *>(
                        stage + p.off_sz + ((mat * 2 + 1) * p.P + rho) * p.sz_box_stride);
                    s_src[mat] = box0 + srow * p.BW + off;
                    z_src[mat] = box1 + srow * p.BW + off;
                }
            }
            // KPS K-blocks per step (the whole stage for one matrix, pairs for
            // gate/up, whose tensor-memory ring is shorter): the step's codes
            // are loaded first, its tensor-memory stores are in flight
            // together, then one wait, then its slots go to the MMA
            constexpr int KPS = kKPS;
#pragma unroll 1
            for (int jp = 0; jp < kStageK / kBlockK; jp += KPS, kbg += KPS) {
                // one wait for the step's tensor-memory slots
                const int stg = kbg / KPS;
                bool got = true;
                if (stg >= kNS) got = tc_wait(&sh.w_empty[stg % kNS], ((stg / kNS) - 1) & 1, abort, false);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                if (warp_live) {
                    uint4 wv[KPS][NMAT];
#pragma unroll
                    for (int e = 0; e < KPS; ++e)
#pragma unroll
                        for (int mat = 0; mat < NMAT; ++mat) {
                            wv[e][mat] = make_uint4(0u, 0u, 0u, 0u);
                            if (row_in_tile)
                                wv[e][mat] = *reinterpret_cast<const uint4 *>(
                                    stage + mat * p.codes_bytes + r * 128 + (((2 * (jp + e) + h) ^ (r & 7)) << 4));
                        }
                    // bf16 constants of each K-block's group, per matrix: (128 + zi)
                    // twice, the scale twice, (zi - z) * scale twice; rows and groups
                    // past the matrix get (128, 0, 0), which dequantizes any code to
                    // 0.  All of the step's constants come first (predicated loads,
                    // no branch between the K-blocks' arithmetic).
                    uint32_t c2[KPS][NMAT], s2[KPS][NMAT], d2[KPS][NMAT];
#pragma unroll
                    for (int e = 0; e < KPS; ++e) {
                        const int gl = chunk_group(c0 + 2 * (jp + e) + h, p.gmagic) - g0;
                        const bool valid = row_valid && g0 + gl <= g_last;
#pragma unroll
                        for (int mat = 0; mat < NMAT; ++mat) {
                            const float sv = valid ? s_src[mat][gl] : 0.0f;
                            const float zv = valid ? z_src[mat][gl] : 0.0f;
                            const float zi = rintf(fminf(fmaxf(zv, 0.0f), 15.0f));
                            c2[e][mat] = bf16x2_pack(128.0f + zi, 128.0f + zi);
                            s2[e][mat] = bf16x2_pack(sv, sv);
                            const float dzs = (zi - zv) * sv;
                            d2[e][mat] = bf16x2_pack(dzs, dzs);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < KPS; ++e) {
                        const int ws = (kbg + e) % kNW;
#pragma unroll
                        for (int mat = 0; mat < NMAT; ++mat) {
                            uint32_t o[16];
                            const uint32_t words[4] = {wv[e][mat].x, wv[e][mat].y, wv[e][mat].z, wv[e][mat].w};
#pragma unroll
                            for (int wi = 0; wi < 4; ++wi) {
                                const uint32_t w = words[wi];
                                const uint32_t t0 = bf16_code_pair(w, magic);
                                const uint32_t t1 = bf16_code_pair(w >> 4, magic);
                                const uint32_t t2 = bf16_code_pair(w >> 8, magic);
                                const uint32_t t3 = bf16_code_pair(w >> 12, magic);
                                o[4 * wi + 0] = bf16x2_fma(bf16x2_sub(t0, c2[e][mat]), s2[e][mat], d2[e][mat]);
                                o[4 * wi + 1] = bf16x2_fma(bf16x2_sub(t1, c2[e][mat]), s2[e][mat], d2[e][mat]);
                                o[4 * wi + 2] = bf16x2_fma(bf16x2_sub(t2, c2[e][mat]), s2[e][mat], d2[e][mat]);
                                o[4 * wi + 3] = bf16x2_fma(bf16x2_sub(t3, c2[e][mat]), s2[e][mat], d2[e][mat]);
                            }
                            tmem_st16(tmem_base + lane_off + w_col(mat, ws) + 16 * h, o);
                        }
                    }
                    tmem_wait_st();
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.w_full[stg % kNS]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[slot]);
            if (++slot == p.S) {
                slot = 0;
                phase ^= 1;
            }
            if (++sir == spr) {
                sir = 0;
                ++tl;
            }
        }
    }

    // =====================================================================
    // MMA warp (one thread issues).
    // =====================================================================
    else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, MP);
            const uint32_t act_s = smem_addr(smem + p.off_act);
            const uint64_t desc_base = smem_desc_sw128(act_s, 1024);
            bool ok = tc_wait(sh.act_ready, 0, abort, false);
            bool any = false;
            int kbg = 0;
            for (int tl = 0; ok && tl < n_tl; ++tl) {
                const int b = tl & 1;
                if (tl >= 2 && !tc_wait(&sh.acc_empty[b], ((tl >> 1) - 1) & 1, abort, false)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // one step (kKPS K-blocks; KBr is a multiple of it) per wait
                // and per commit
                for (int kb0 = 0; kb0 < KBr; kb0 += kKPS, kbg += kKPS) {
                    const int stg = kbg / kKPS;
                    if (!tc_poll(&sh.w_full[stg % kNS], (stg / kNS) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll
                    for (int e = 0; e < kKPS; ++e) {
                        const int kb = kb0 + e;
                        const int ws = (kbg + e) % kNW;
                        // descriptors advance by whole 16-byte units: one add per MMA
                        const uint64_t bdesc0 = desc_base + (uint64_t)((uint32_t)kb * (MP * 128) >> 4);
#pragma unroll
                        for (int mat = 0; mat < NMAT; ++mat) {
                            const uint32_t a0 = tmem_base + w_col(mat, ws);
                            const uint32_t d = tmem_base + acc_col(mat, b);
#pragma unroll
                            for (int jj = 0; jj < kBlockK / 16; ++jj)
                                tc_mma_ts(d, a0 + 8 * jj, bdesc0 + (uint64_t)(2 * jj), idesc,
                                          (kb | jj) != 0 ? 1u : 0u);
                        }
                    }
                    any = true;
                    tc_commit(&sh.w_empty[stg % kNS]);
                }
                if (!ok) break;
                tc_commit(&sh.acc_full[b]);
            }
            if (!ok && any) {
                // let the MMAs in flight finish before tensor memory is freed
                tc_commit(sh.drain);
                tc_drain_wait(sh.drain, 0);
            }
        }
        __syncwarp();
    }

    // =====================================================================
    // Epilogue warps: accumulator -> (cluster split-K sum) -> outputs.
    // =====================================================================
    else {
        const int et = threadIdx.x - kEpBase;  // 0..127
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        float *red = reinterpret_cast<float *>(smem + p.off_red);
        // A thread whose wait fails keeps walking the loop (skipping work) so
        // that the group's named barriers are always reached by all 128.
        bool ok = true;
        if (ks > 1) cluster_wait();
        cwaited = true;
        // the norm prologue's inverse RMS per lane (1 without the prologue)
        float *s_inv = reinterpret_cast<float *>(smem + p.off_misc + 256);
        if constexpr (NORM) {
            // every rank's square sums (rank order), then 1 / sqrt(mean + eps)
            ok = __all_sync(0xffffffffu, tc_wait(sh.norm_full, 0, abort, true));
            if (et < p.M) {
                float total = 0.0f;
                if (ok) {
                    for (int j = 0; j < ks; ++j) total += dsmem_ld_f32(dsmem_addr(smem_addr(&sh.part[et]), j));
                }
                s_inv[et] = 1.0f / sqrtf(total / (float)p.K + p.eps);
            }
            named_barrier(2, kEpWarps * 32);
            // norm_out = (x * inv) * W_norm in f32 from x recomputed, each
            // 8-code chunk of a lane written once over the clusters: chunk c
            // of lane m of this rank's K range by cluster (m * n_chunks + c)
            // mod n_clusters
            if (ok && p.norm_out) {
                const int n_chunks = KBr * 8;
                const int k_base = st0 * kStageK;
                for (int idx = et; idx < p.M * n_chunks; idx += kEpWarps * 32) {
                    const int m = idx / n_chunks;
                    const int c = idx - m * n_chunks;
                    const int k = k_base + 8 * c;
                    if (k >= p.K || (m * n_chunks + c) % p.n_clusters != cid) continue;
                    const size_t o = (size_t)m * p.K + k;
                    const float4 *a4 = reinterpret_cast<const float4 *>(p.A + o);
                    const float4 *w4 = reinterpret_cast<const float4 *>(p.W_norm + k);
                    float4 x0 = __ldg(a4), x1 = __ldg(a4 + 1);
                    if (p.A_b) {
                        const float4 *b4 = reinterpret_cast<const float4 *>(p.A_b + o);
                        const float4 b0 = __ldg(b4), b1 = __ldg(b4 + 1);
                        x0.x += b0.x; x0.y += b0.y; x0.z += b0.z; x0.w += b0.w;
                        x1.x += b1.x; x1.y += b1.y; x1.z += b1.z; x1.w += b1.w;
                    }
                    const float4 g0 = __ldg(w4), g1 = __ldg(w4 + 1);
                    const float iv = s_inv[m];
                    float4 *no = reinterpret_cast<float4 *>(p.norm_out + o);
                    no[0] = make_float4((x0.x * iv) * g0.x, (x0.y * iv) * g0.y, (x0.z * iv) * g0.z,
                                        (x0.w * iv) * g0.w);
                    no[1] = make_float4((x1.x * iv) * g1.x, (x1.y * iv) * g1.y, (x1.z * iv) * g1.z,
                                        (x1.w * iv) * g1.w);
                }
            }
        }
        for (int tl = 0; tl < n_tl; ++tl) {
            const int b = tl & 1;
            // every outcome is made warp-uniform: the tensor-memory loads are
            // collective
            ok = __all_sync(0xffffffffu, ok && tc_wait(&sh.acc_full[b], (tl >> 1) & 1, abort, false));
            // accumulator -> this CTA's partial tile in shared memory, 16
            // columns at a time: red[mat][lane m][row r]
            if (tl >= 1 && ks > 1)
                ok = __all_sync(0xffffffffu, ok && tc_wait(sh.red_empty, (tl - 1) & 1, abort, true));
            if (ok) {
                tc_fence_after_sync();
#pragma unroll
                for (int mat = 0; mat < NMAT; ++mat) {
#pragma unroll
                    for (int c = 0; c < MP / 16; ++c) {
                        uint32_t u[16];
                        tmem_ld16(tmem_base + lane_off + acc_col(mat, b) + 16 * c, u);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) red[(mat * MP + 16 * c + e) * 128 + r] = __uint_as_float(u[e]);
                    }
                }
                tc_fence_before_sync();
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&sh.acc_empty[b]);
            const int row0 = (cid + tl * p.n_clusters) * p.TR;
            if (ks == 1) {
                // the thread reads back only what it wrote (its row)
                const int col = row0 + r;
                if (ok && r < p.TR && col < p.N) {
                    for (int m = 0; m < p.M; ++m) {
                        const float iv = NORM ? s_inv[m] : 1.0f;
                        store_out<EPI>(p, m, col, red[m * 128 + r] * iv,
                                       red[((NMAT - 1) * MP + m) * 128 + r] * iv);
                    }
                }
                continue;
            }
            // split-K: every rank sums its share of the rows over all ranks,
            // in rank order
            named_barrier(2, kEpWarps * 32);
            if (et == 0) {
                // the group's partial-tile writes (ordered by the barrier) are
                // released to the peers at cluster scope
                fence_acq_rel_cluster();
                for (int j = 0; j < ks; ++j) mbar_arrive_cluster(dsmem_addr(smem_addr(sh.red_full), j));
            }
            ok = __all_sync(0xffffffffu, ok && tc_wait(sh.red_full, tl & 1, abort, true));
            if (ok) {
                // this rank's share: whole groups of 4 rows; per group and lane,
                // every rank's 16-byte partial is loaded before the rank-order sum
                const int g4 = p.TR / 4;
                const int q0 = 4 * (g4 * rank / ks);
                const int q1 = 4 * (g4 * (rank + 1) / ks);
                const int n4 = (q1 - q0) / 4;
                const uint32_t red_s = smem_addr(red);
                for (int idx = et; idx < n4 * p.M; idx += kEpWarps * 32) {
                    const int m = idx / n4;
                    const int rr = q0 + 4 * (idx - m * n4);
                    float4 sum[NMAT];
#pragma unroll
                    for (int mat = 0; mat < NMAT; ++mat) {
                        const uint32_t off = (uint32_t)(((mat * MP + m) * 128 + rr) * 4);
                        float4 part[kMaxKs];
#pragma unroll
                        for (int j = 0; j < kMaxKs; ++j)
                            if (j < ks) part[j] = dsmem_ld_f32x4(dsmem_addr(red_s + off, j));
                        float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                        for (int j = 0; j < kMaxKs; ++j) {
                            if (j < ks) {
                                a.x += part[j].x;
                                a.y += part[j].y;
                                a.z += part[j].z;
                                a.w += part[j].w;
                            }
                        }
                        sum[mat] = a;
                    }
                    const float g[4] = {sum[0].x, sum[0].y, sum[0].z, sum[0].w};
                    const float u4[4] = {sum[NMAT - 1].x, sum[NMAT - 1].y, sum[NMAT - 1].z, sum[NMAT - 1].w};
                    const float iv = NORM ? s_inv[m] : 1.0f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = row0 + rr + e;
                        if (rr + e < p.TR && col < p.N) store_out<EPI>(p, m, col, g[e] * iv, u4[e] * iv);
                    }
                }
            }
            named_barrier(2, kEpWarps * 32);
            if (et == 0) {
                for (int j = 0; j < ks; ++j) mbar_arrive_cluster(dsmem_addr(smem_addr(sh.red_empty), j));
            }
        }
        // every peer has finished reading this CTA's last partial tile
        if (ks > 1 && n_tl > 0) (void)tc_wait(sh.red_empty, (n_tl - 1) & 1, abort, true);
    }

    // ---- teardown ----
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
    if (ks > 1) {
        if (!cwaited) cluster_wait();
        cluster_sync_all();  // no peer reads this CTA's shared memory any more
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

struct TcPlan {
    int ks, TR, n_tiles, n_clusters, S, gps;
    uint32_t smem;
};

// Shared-memory layout of one ring stage: packed codes of every matrix
// (TR rows x 128 bytes each), then per matrix and array (scale, zero) and row
// residue one box of TR/P super-rows x BW floats, then the tail rows.
struct StageGeom {
    int P, BW;
    uint32_t codes_bytes, sz_box_bytes, sz_box_stride, off_sz, off_tail, stage_bytes;
};

StageGeom stage_geom(int TR, int nmat, int G, int gps)
{
    StageGeom g;
    g.P = 4 / gcd_int(G, 4);                    // P rows of G floats: a 16-byte multiple
    g.BW = (3 + gps + 3) / 4 * 4;                // a stage's groups from a 16-byte aligned start
    g.codes_bytes = (uint32_t)TR * 128u;
    g.sz_box_bytes = (uint32_t)(TR / g.P) * (uint32_t)g.BW * 4u;
    g.sz_box_stride = (g.sz_box_bytes + 127u) / 128u * 128u;
    g.off_sz = (uint32_t)nmat * g.codes_bytes;
    g.off_tail = g.off_sz + (uint32_t)nmat * 2u * (uint32_t)g.P * g.sz_box_stride;
    const uint32_t tail = (uint32_t)nmat * 2u * 4u * (uint32_t)g.BW * 4u;
    g.stage_bytes = (g.off_tail + tail + 1023u) / 1024u * 1024u;
    return g;
}

constexpr int kMaxDevices = 64;

// Co-resident clusters of `ks` one-CTA-per-SM blocks (queried once per device).
int max_clusters(int dev, int ks, const void *kern)
{
    static std::atomic<int> cache[kMaxDevices][9];
    static std::once_flag init_flag;
    std::call_once(init_flag, []() {
        for (int d = 0; d < kMaxDevices; ++d)
            for (int k = 0; k < 9; ++k) cache[d][k].store(-1);
    });
    if (dev < 0 || dev >= kMaxDevices || ks < 1 || ks > 8) return 0;
    int v = cache[dev][ks].load(std::memory_order_acquire);
    if (v >= 0) return v;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cfg.gridDim = dim3((unsigned)(sms / ks * ks > 0 ? sms / ks * ks : ks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 200u * 1024u;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    cache[dev][ks].store(n, std::memory_order_release);
    return n;
}

bool plan_tc(const Call &call, int MP, int dev, const void *kern, int smem_optin, TcPlan &best)
{
    const int n_st = (call.K + kStageK - 1) / kStageK;
    const int gps = groups_per_stage(call.gs, kStageK);
    if (gps > kMaxGps) return false;
    const int nmat = call.nmat;
    double best_cost = 0.0;
    bool found = false;
    for (int ks = 1; ks <= 8 && ks <= n_st; ++ks) {
        const int clusters_max = max_clusters(dev, ks, kern);
        if (clusters_max <= 0) continue;
        const int spr_max = (n_st + ks - 1) / ks;
        const uint32_t act = (uint32_t)spr_max * (kStageK / kBlockK) * MP * 128u;
        const uint32_t red = (uint32_t)nmat * MP * 128u * 4u;
        for (int TR = 128; TR >= 16; TR -= 8) {
            const uint32_t stage = stage_geom(TR, nmat, call.K / call.gs, gps).stage_bytes;
            const uint32_t fixed = 1024u + act + round_up(red, 1024u) + 1024u;
            if (fixed + 2u * stage > (uint32_t)smem_optin) continue;
            int S = (int)(((uint32_t)smem_optin - fixed) / stage);
            if (S > kMaxStages) S = kMaxStages;
            const int n_tiles = (call.N + TR - 1) / TR;
            const int clusters = n_tiles < clusters_max ? n_tiles : clusters_max;
            const int waves = (n_tiles + clusters - 1) / clusters;
            // critical-path work of one CTA, in codes: its tiles' share of K,
            // the per-tile pipeline fill and epilogue, and the activation staging
            // (staging: the lanes' f32 activations of the K range, read at
            // roughly 100 GB/s per SM, against ~75 G codes/s of dequant)
            const double per_tile = (double)TR * spr_max * kStageK * nmat + 49152.0 * nmat;
            const double staging = 0.77 * (double)spr_max * kStageK * call.M * 4.0 * (call.norm ? 2.0 : 1.0);
            const double cost = waves * per_tile + staging;
            if (!found || cost < best_cost * 0.999) {
                found = true;
                best_cost = cost;
                best.ks = ks;
                best.TR = TR;
                best.n_tiles = n_tiles;
                best.n_clusters = clusters;
                best.S = S;
                best.gps = gps;
                uint32_t smem = fixed + (uint32_t)S * stage;
                best.smem = smem < kMinSmem ? kMinSmem : smem;
            }
        }
    }
    return found;
}

template <int MP, int NMAT, bool NORM, int EPI>
cudaError_t launch_tc_variant(const Call &call, cudaStream_t stream)
{
    auto kern = tc_matvec_kernel<MP, NMAT, NORM, EPI>;
    int dev = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    int optin = 0;
    if ((err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return err;
    // the 1024-byte alignment pad is part of every plan
    static std::atomic<unsigned char> ready[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices || !ready[dev].load(std::memory_order_acquire)) {
        if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin)) != cudaSuccess)
            return err;
        if (dev >= 0 && dev < kMaxDevices) ready[dev].store(1, std::memory_order_release);
    }
    TcPlan pl{};
    if (!plan_tc(call, MP, dev, reinterpret_cast<const void *>(kern), optin, pl)) return cudaErrorInvalidValue;

    TcParams prm{};
    EncodeTiledFn encode = encode_tiled_fn();
    if (!encode) return cudaErrorNotSupported;
    for (int mat = 0; mat < NMAT; ++mat) {
        const cuuint64_t dims[2] = {(cuuint64_t)(call.K / 8), (cuuint64_t)call.N};
        const cuuint64_t strides[1] = {(cuuint64_t)call.K / 2};
        const cuuint32_t box[2] = {32u, (cuuint32_t)pl.TR};
        const cuuint32_t estr[2] = {1u, 1u};
        if (encode(&prm.codes[mat], CU_TENSOR_MAP_DATA_TYPE_UINT32, 2,
                   const_cast<uint32_t *>(call.Bq[mat]), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // scales / zeros as [Q][P*G] super-rows (row stride a 16-byte multiple)
        const int P = 4 / gcd_int(call.K / call.gs, 4);
        const int G = call.K / call.gs;
        const int BW = (3 + pl.gps + 3) / 4 * 4;
        const cuuint64_t dims[2] = {(cuuint64_t)P * G, (cuuint64_t)(call.N / P)};
        const cuuint64_t strides[1] = {(cuuint64_t)P * G * 4u};
        const cuuint32_t box[2] = {(cuuint32_t)BW, (cuuint32_t)(pl.TR / P)};
        const cuuint32_t estr[2] = {1u, 1u};
        for (int mat = 0; mat < NMAT; ++mat)
            for (int arr = 0; arr < 2; ++arr) {
                const float *base = arr == 0 ? call.scales[mat] : call.zeros[mat];
                if (encode(&prm.sz[mat][arr], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                    return cudaErrorInvalidValue;
            }
    }
    prm.M = call.M;
    prm.K = call.K;
    prm.N = call.N;
    prm.gs = call.gs;
    prm.G = call.K / call.gs;
    prm.TR = pl.TR;
    prm.n_tiles = pl.n_tiles;
    prm.n_clusters = pl.n_clusters;
    prm.ks = pl.ks;
    prm.n_st = (call.K + kStageK - 1) / kStageK;
    prm.S = pl.S;
    prm.gps = pl.gps;
    const int spr_max = (prm.n_st + pl.ks - 1) / pl.ks;
    const StageGeom sg = stage_geom(pl.TR, NMAT, prm.G, pl.gps);
    prm.P = sg.P;
    prm.logP = sg.P == 1 ? 0 : sg.P == 2 ? 1 : 2;
    prm.Q = call.N / sg.P;
    {
        const unsigned long long d = (unsigned long long)(call.gs / 32);
        prm.gmagic = ((1ull << 40) + d - 1) / d;
    }
    prm.BW = sg.BW;
    prm.codes_bytes = sg.codes_bytes;
    prm.sz_box_bytes = sg.sz_box_bytes;
    prm.sz_box_stride = sg.sz_box_stride;
    prm.off_sz = sg.off_sz;
    prm.off_tail = sg.off_tail;
    prm.stage_bytes = sg.stage_bytes;
    prm.off_act = 0;
    const uint32_t act = (uint32_t)spr_max * (kStageK / kBlockK) * MP * 128u;
    const uint32_t red = (uint32_t)NMAT * MP * 128u * 4u;
    prm.off_ring = round_up(act, 1024u);
    prm.off_red = prm.off_ring + (uint32_t)pl.S * prm.stage_bytes;
    prm.off_misc = prm.off_red + round_up(red, 1024u);
    prm.off_bar = prm.off_misc + 384u;  // part[32], tensor-memory base, abort flag, inv[32]
    if (prm.off_bar + 80u * 8u + 1024u > pl.smem) return cudaErrorInvalidValue;
    prm.magic_bf16 = 0x43004300u;
    prm.A = call.A;
    if (call.norm) {
        prm.A_b = call.norm->A_b;
        prm.W_norm = call.norm->W_norm;
        prm.eps = call.norm->eps;
        prm.residual_out = call.norm->residual_out;
        prm.norm_out = call.norm->norm_out;
    }
    for (int mat = 0; mat < 2; ++mat) {
        const int src = mat < call.nmat ? mat : 0;
        prm.scales[mat] = call.scales[src];
        prm.zeros[mat] = call.zeros[src];
    }
    for (int i = 0; i < 4; ++i) {
        prm.out[i] = call.out[i];
        prm.seg_start[i] = call.seg_start[i];
        prm.seg_len[i] = call.seg_len[i];
    }

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3((unsigned)(pl.n_clusters * pl.ks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pl.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic stream serialization: the CTAs may start while the
    // previous kernel in the stream finishes (the producer streams weights at
    // once); the dequant warps wait for that kernel's completion
    // (griddepcontrol.wait) before reading activations.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if ((err = cudaLaunchKernelEx(&cfg, kern, prm)) != cudaSuccess) return err;
    return cudaGetLastError();
}

template <int MP>
cudaError_t dispatch_tc(const Call &call, cudaStream_t stream)
{
    const bool norm = call.norm != nullptr;
    switch (call.epi) {
    case kEpiStore:
        return norm ? launch_tc_variant<MP, 1, true, kEpiStore>(call, stream)
                    : launch_tc_variant<MP, 1, false, kEpiStore>(call, stream);
    case kEpiQuad:
        return launch_tc_variant<MP, 1, false, kEpiQuad>(call, stream);
    case kEpiGated:
        return norm ? launch_tc_variant<MP, 2, true, kEpiGated>(call, stream)
                    : launch_tc_variant<MP, 2, false, kEpiGated>(call, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace

bool tc_path_supported(const Call &call)
{
    if (call.M < 16 || call.M > 32) return false;
    // gated inputs and the dual projection run on the CUDA-core kernels
    if (call.gate_kind != kGateNone || call.epi == kEpiDual) return false;
    // scales and zeros are read by tensor-map copies of whole super-rows of
    // P = 4 / gcd(G, 4) rows (16-byte aligned bases, at least one super-row)
    const int P = 4 / gcd_int(call.K / call.gs, 4);
    if (call.N < P) return false;
    for (int m = 0; m < call.nmat; ++m) {
        if ((reinterpret_cast<uintptr_t>(call.scales[m]) & 15u) != 0) return false;
        if ((reinterpret_cast<uintptr_t>(call.zeros[m]) & 15u) != 0) return false;
    }
    if (groups_per_stage(call.gs, kStageK) > kMaxGps) return false;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
    return major == 10 && minor == 3 && encode_tiled_fn() != nullptr;
}

cudaError_t launch_tc(const Call &call, cudaStream_t stream)
{
    // fewer than 16 lanes (row chunks of a GEMM) run padded to 16
    return call.M <= 16 ? dispatch_tc<16>(call, stream) : dispatch_tc<32>(call, stream);
}

bool tc_rows_supported(const Call &call)
{
    if (call.M < 1 || call.M > 32) return false;
    Call c = call;
    c.M = 16;  // every other condition as for 16 lanes
    return tc_path_supported(c);
}

cudaError_t read_tc_device_error(unsigned int *bits, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(bits, g_tc_error, sizeof(unsigned int));
    if (err != cudaSuccess || !clear) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(unsigned int));
}

}  // namespace gq4

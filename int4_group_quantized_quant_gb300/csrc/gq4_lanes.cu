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
//     A shift by 8 brings the other four codes of the word to the same places:
//     five integer operations decode a word (8 codes).
//   * Activations are staged per lane and 128-code block as 22-bit fixed-point
//     integers X = rint(x 2^k) (the block's largest magnitude in [2^21, 2^22])
//     split into X = 2048 h + l, both exact in fp16; the odd code positions
//     take h / 16 and l / 16, matching the 16 q of their codes.
//   * mma.sync m16n8k16 (fp16 inputs, f32 accumulation): 16 weight columns
//     (rows of the MMA) times 8 columns of B = {h, l} of 4 lanes.  Every
//     product and partial sum is an integer times 2^-24 below 2^24 of them,
//     so the block's sums of q h and q l are exact; zi (sum h) and zi (sum l)
//     come off exactly (zi the integer part of the zero point: codes equal to
//     an integer zero give exactly nothing).
//   * Per block, column and lane: y += s * (2^(24-k) (2048 H + L) - (z - zi)
//     S), with H and L the exact sums of (q - zi) h and (q - zi) l and S the
//     f32 sum of the block's activations (the fractional part of the zero
//     comes off through S).
//
// Decomposition:
//   * Persistent grid of thread-block clusters, one CTA per SM; 16 consumer
//     warps, a producer warp, a helper warp and a scale warp per CTA.  Two
//     cluster forms:
//     - CTA pairs (K up to 32 blocks, at most 32 groups): each CTA owns a
//       contiguous range of whole columns and stages half of K's activations,
//       storing them into its own and its partner's shared memory;
//     - split K (longer K): the 2-4 CTAs of a cluster own the same columns,
//       each a chunk of whole scale groups of K, and rank 0 adds the others'
//       per-stage partial sums (sent through distributed shared memory) in
//       rank order before the epilogue.
//   * The producer streams the codes through a ring of S stages.  A stage is
//     one MMA tile: 16 columns (8 gate and 8 up columns for gate/up, 8 and 8
//     of the two matrices for dual), fetched as bulk copies (two runs of 8
//     whole columns, or one copy per column chunk when K is split) into two
//     regions whose bases differ by 64 bytes mod 128, so that MMA rows g and
//     g + 1 (lanes 4g.. and 4g+4..) read disjoint bank halves.  Stages beyond
//     the ring are prefetched into L2.
//   * A scale warp fills each stage's scale scratch ({s, z} per MMA row and
//     group, laid out for conflict-free reads) by 16-, 8- or 4-byte cp.async
//     straight from global memory as soon as the ring entry is free,
//     completing on the stage's mbarrier, so that no warp waits for the
//     scales' round trip under the weight stream.
//   * The helper warp adds each stage's 16 partial sums in warp order,
//     applies the norm's inverse RMS and the epilogue, and writes the
//     outputs.
//   * The consumer warps split each stage's K into 16 slices of whole 128-code
//     blocks (at most 2 per warp, held in registers as MMA B fragments); per
//     stage a warp waits for the codes and the scratch, runs its blocks,
//     releases the ring entry and posts its partials to a 2-deep partial
//     ring (once the helper has read stage i - 2's from it).  96 registers a
//     thread: 19 warps put 5 on a scheduler.
//   * Programmatic dependent launch as in the one-lane kernel: the producer
//     reads weights (codes, scales) before the dependency wait, the consumers
//     wait before reading activations; a kernel signals its dependents at its
//     last stage.
//   * Every mbarrier wait is bounded in time; on expiry the kernel records an
//     error in a device word (gq4_device_error), writes NaN and releases its
//     stages.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "gq4_device.cuh"
#include "gq4_host.h"
#include "gq4_internal.h"
#include "gq4_onelane.cuh"
#include "gq4_tma.cuh"

namespace gq4 {

// Sticky device-side error word of this path (bit 5: a wait timed out).
__device__ unsigned int g_lanes_error = 0;

namespace {

constexpr int kConsumerWarps = 16;
constexpr int kProducerWarp = kConsumerWarps;      // bulk copies of the codes
constexpr int kHelperWarp = kConsumerWarps + 1;    // cross-warp sums, outputs
constexpr int kScaleWarp = kConsumerWarps + 2;     // scale scratch copies
constexpr int kThreads = (kConsumerWarps + 3) * 32;
constexpr int kBar2Threads = (kConsumerWarps + 1) * 32;  // consumers + producer
constexpr int kCT = kConsumerWarps * 32;
// registers per thread: 19 warps put 5 on a scheduler, 5 * 32 * 96 <= 16384
constexpr int kMaxRegs = 96;
constexpr int kMaxStages = 16;
constexpr int kBlock = 128;  // codes per activation block (one scale exponent, one MMA run)
constexpr int kPrefetchAhead = 16;  // stages prefetched into L2 ahead of the ring copies
constexpr int kPreStages = 3;       // stages issued before the consumers' activation loads return
constexpr int kMaxWarpBlocks = 2;   // 128-code blocks per consumer warp (K <= 4096 in one CTA)
constexpr int kMaxSplit = 4;        // K chunks per cluster when K is split
constexpr int kCombine = 4;         // stages of partial sums in flight to a cluster's rank 0
constexpr int kPartRing = 2;        // stages of consumer partial sums awaiting the helper
constexpr int kSplitWarpBlocks = 2; // preferred blocks per consumer warp when K is split
constexpr uint32_t kSmemLimit = 226u * 1024u;  // of the 227 KB a block may opt in to

// First scale group of K chunk r of ks (r = ks: G).  Inner bounds fall on
// multiples of 4 groups when G is, else of 2 when G is even, so that the
// chunk's scale rows start 16- (8-) byte aligned for the scale copies.
__host__ __device__ __forceinline__ int chunk_group(int G, int ks, int r)
{
    if (r >= ks) return G;
    const int a = (G & 3) == 0 ? 4 : (G & 1) == 0 ? 2 : 1;
    return (int)((long long)G * r / ks) / a * a;
}

struct LanesParams {
    int M, K, N, gs;
    int KW;          // packed words per column (K / 8)
    int KB;          // 128-code blocks per column
    int G;           // scale groups per column
    int bpg;         // blocks per scale group (gs / 128, a power of two)
    int bpg_shift;   // log2(bpg)
    int S;           // ring depth
    int ks;          // K chunks per cluster (1: CTA pairs share the staging of all of K)
    int Gs;          // scale groups per ring entry's scratch (G, or the largest chunk's)
    int unit;        // column granularity of the balanced split
    int n_units;
    uint32_t stage_bytes;
    uint32_t off_act, off_fx, off_part, off_scr, off_misc, off_cmb, off_bar;
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

// Cluster helpers (CTA pairs share the activation staging).
__device__ __forceinline__ uint32_t lanes_cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared-memory address of the same location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t lanes_mapa(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Every thread of the cluster arrives once (split barrier: arrive, later wait).
__device__ __forceinline__ void lanes_cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void lanes_cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stores into a peer CTA's shared memory that complete on its mbarrier's
// transaction count (addresses from lanes_mapa).
__device__ __forceinline__ void st_async_v2(uint32_t raddr, uint32_t a, uint32_t b, uint32_t rbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];"
                 ::"r"(raddr), "r"(a), "r"(b), "r"(rbar) : "memory");
}

__device__ __forceinline__ void st_async_v4(uint32_t raddr, float4 v, uint32_t rbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(raddr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar) : "memory");
}

__device__ __forceinline__ void st_async_f32(uint32_t raddr, float v, uint32_t rbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
                 ::"r"(raddr), "f"(v), "r"(rbar) : "memory");
}

// 4-byte asynchronous copy global -> shared (both 4-byte aligned).
__device__ __forceinline__ void lanes_cp_async_4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// 8-byte asynchronous copy global -> shared (both 8-byte aligned) of the
// first `bytes` (4 or 8) of the source; a short copy zero-fills the rest.
__device__ __forceinline__ void lanes_cp_async_8(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(bytes)
                 : "memory");
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned) of the
// first `bytes` (4..16) of the source; the rest of the 16 destination bytes
// are zero-filled.
__device__ __forceinline__ void lanes_cp_async_16(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(bytes)
                 : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (counted in the barrier's expected arrivals).
__device__ __forceinline__ void lanes_cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive on an mbarrier of a CTA of the cluster (address from lanes_mapa).
__device__ __forceinline__ void lanes_remote_arrive(uint32_t rbar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar) : "memory");
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

// Bulk prefetch of global memory into L2 (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
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

__device__ __forceinline__ uint32_t h2_bits(__half2 h)
{
    return *reinterpret_cast<uint32_t *>(&h);
}

// Reduce-scatter of U values per lane (U = 4, 8 or 16) over the 32 lanes of
// a warp: afterwards lane l holds the reduction of unit (l / (32/U)) over all
// 32 lanes, as do the other 32/U - 1 lanes of its run (unit u's run starts at
// lane 32u/U).  A fixed order of operations, so the result is the same
// whatever the units hold.
template <int U>
__device__ __forceinline__ int rs_unit(int lane)
{
    return lane / (32 / U);
}

template <int U>
__device__ __forceinline__ int rs_owner(int u)
{
    return u * (32 / U);
}

template <int U, class T, class Op>
__device__ __forceinline__ T reduce_scatter(const T (&v)[U], int lane, Op op)
{
    static_assert(U == 4 || U == 8 || U == 16, "units per warp");
    T a[U];
#pragma unroll
    for (int i = 0; i < U; ++i) a[i] = v[i];
    int n = U;
#pragma unroll
    for (int off = 16; off >= 32 / U; off >>= 1) {
        n >>= 1;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < U / 2; ++i) {
            if (i >= n) break;
            const T keep = up ? a[i + n] : a[i];
            const T send = up ? a[i] : a[i + n];
            a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
        }
    }
#pragma unroll
    for (int off = 16 / U; off >= 1; off >>= 1) a[0] = op(a[0], __shfl_xor_sync(0xffffffffu, a[0], off));
    return a[0];
}

struct OpAdd {
    template <class T>
    __device__ __forceinline__ T operator()(T x, T y) const { return x + y; }
};
struct OpMax {
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y) const { return max(x, y); }
};

constexpr int kBadScale = 1 << 20;  // the scale exponent of a block holding an inf or NaN

// Scale of a block from its largest magnitude as bits (an inf or NaN compares
// above any finite): X = rint(x 2^k) puts the largest magnitude in
// [2^21, 2^22]; f = 2^(24 - k) turns the MMA's sums (units of 2^-24) back
// into activation units.  A non-finite block gives k = kBadScale and f = NaN.
__device__ __forceinline__ void block_scale(uint32_t mb, int &k, float &f)
{
    k = 0;
    f = 0.0f;
    if (mb >= 0x7f800000u) {
        k = kBadScale;
    } else if (mb != 0u) {
        int E = ilogbf(__uint_as_float(mb));  // the largest magnitude in [2^E, 2^(E+1))
        if (E > 124) {
            k = kBadScale;  // 2^(24-k) would leave the f32 range
        } else {
            E = E < -129 ? -129 : E;  // subnormal activations: a smaller scale
            k = 21 - E;
            f = pow2i(3 + E);
        }
    }
    if (k == kBadScale) f = __int_as_float(0x7fffffff);  // the block's lane results become NaN
}

// Two integers as fp16 halves: a, and b / 16 (exact).
__device__ __forceinline__ uint32_t piece_pair(int a, int b)
{
    return h2_bits(__floats2half2_rn((float)a, (float)b * 0.0625f));
}

template <int V>
using IntC = std::integral_constant<int, V>;

// NP: lanes per MMA (2 or 4; the N columns are {hi, lo} of each lane).
// SPLIT: K split over the cluster (p.ks > 1), else CTA pairs.
template <int NMAT, int PRO, int EPI, int NP, bool SPLIT>
__global__ void __maxnreg__(kMaxRegs) lanes_matvec_kernel(const __grid_constant__ LanesParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);  // codes of a stage landed
    uint64_t *empty = full + kMaxStages;   // the consumer warps are done with a ring entry
    uint64_t *sfull = empty + kMaxStages;  // a ring entry's scale scratch landed
    uint64_t *pbar = sfull + kMaxStages;   // the consumer warps wrote a ring entry's partials
    uint64_t *pfree = pbar + kMaxStages;   // the helper has read a ring entry's partials
    uint64_t *aload = pfree + kMaxStages;  // the consumer warps' activation loads returned
    uint64_t *peerb = aload + 1;           // the partner CTA's half of the staging landed
    uint64_t *cfull = peerb + 1;           // [kCombine] split K: the other ranks' partials landed
    uint64_t *cfree = cfull + kCombine;    // [kCombine] split K: rank 0 has read a combine entry
    int *s_seq = reinterpret_cast<int *>(cfree + kCombine);  // stage a ring entry holds
    float *s_inv = reinterpret_cast<float *>(smem + p.off_misc);        // [4] inverse RMS per lane
    float *s_sq = s_inv + 4;                                            // [warps][4] square sums
    // [kMaxSplit - 1][4] the other CTAs' square sums (pairs: the partner's half in [0])
    float *s_sqp = s_sq + 4 * kConsumerWarps;
    unsigned char *s_act = smem + p.off_act;
    const float4 *s_fx = reinterpret_cast<const float4 *>(smem + p.off_fx);  // [KB][4] {f1, f2, X, 0}

    constexpr int TCOLS = NMAT == 2 ? 8 : 16;  // output columns per stage
    constexpr bool NORM = PRO == kProNorm;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Two cluster forms.  CTA pairs (ks = 1): each CTA owns its columns and
    // stages half of K's activations for both.  Split K (ks > 1): the ks CTAs
    // of a cluster own the same columns, each a chunk of whole scale groups
    // of K, and rank 0 adds the others' partial sums in rank order.
    constexpr bool split = SPLIT;
    const uint32_t crank = lanes_cluster_rank();
    const int owner = split ? (int)blockIdx.x / p.ks : (int)blockIdx.x;
    const int n_owners = split ? (int)gridDim.x / p.ks : (int)gridDim.x;
    const int u0 = (int)((long long)p.n_units * owner / n_owners);
    const int u1 = (int)((long long)p.n_units * (owner + 1) / n_owners);
    const int col_begin = u0 * p.unit;
    const int col_end = min(u1 * p.unit, p.N);
    // a CTA without columns still stages its half of the activations for
    // its partner (and then runs no stage)
    const int ncols = col_end > col_begin ? col_end - col_begin : 0;
    const int n_stages = (ncols + TCOLS - 1) / TCOLS;
    // this CTA's groups [g_lo, g_lo + GL) and blocks [kbc0, kbc0 + KBL) of K
    const int g_lo = split ? chunk_group(p.G, p.ks, (int)crank) : 0;
    const int GL = split ? chunk_group(p.G, p.ks, (int)crank + 1) - g_lo : p.G;
    const int kbc0 = g_lo * p.bpg;
    const int KBL = GL * p.bpg;
    const uint32_t cb = (uint32_t)KBL * 64u;  // a column's codes in a stage (bytes)
    const uint32_t off_reg1 = 8u * cb + 64u;  // second region of a stage (64 mod 128)
    // the blocks [kb_lo, kb_hi) of the chunk this CTA stages (pairs: its half,
    // the partner the rest)
    const uint32_t peer = crank ^ 1u;
    const int kb_half = KBL / 2;
    const int kb_lo = split ? 0 : (crank ? kb_half : 0);
    const int kb_hi = split ? KBL : (crank ? KBL : kb_half);
    const int kb_peer = split ? 0 : (crank ? kb_half : KBL - kb_half);  // blocks the partner stages

    // =====================================================================
    // Producer warp: lane 0 the bulk copies of the codes and the L2
    // prefetches.
    // =====================================================================
    if (warp == kProducerWarp) {
        if (lane == 0) {
            for (int s = 0; s < p.S; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kConsumerWarps);
                mbar_init(&sfull[s], 32);  // the scale warp lanes' cp.async arrivals
                s_seq[s] = -1;
            }
            for (int s = 0; s < kPartRing; ++s) {
                mbar_init(&pbar[s], kConsumerWarps);
                mbar_init(&pfree[s], 1);
            }
            mbar_init(aload, kConsumerWarps);
            mbar_init(peerb, 1);  // completed by the partner's stores and one local expect
            for (int s = 0; s < kCombine; ++s) {
                mbar_init(&cfull[s], 1);  // rank 0's expect plus the other ranks' stores
                mbar_init(&cfree[s], 1);  // rank 0's remote arrive
            }
            mbar_fence_init();
        }
        __syncwarp();
        lanes_cluster_arrive();  // after the initialisation: the cluster may now use peerb, cfull, cfree
        lanes_bar_arrive(4, kBar2Threads);  // the consumers' first mbarrier use (aload)
        lanes_bar_arrive(2, kBar2Threads);  // the consumers' barrier after their prologue
        lanes_bar_arrive(3, 96);            // the helper's and the scale warp's
        {
            int issued = 0;
            bool ok = true;
            // the codes of stage i as (first column, count) per region
            auto stage_regions = [&](int i, int (&rc)[2], int (&rn)[2]) {
                const int c0 = col_begin + i * TCOLS;
                const int nc = min(TCOLS, col_end - c0);
                if constexpr (NMAT == 2) {
                    rc[0] = rc[1] = c0;
                    rn[0] = rn[1] = nc;
                } else {
                    rc[0] = c0;
                    rn[0] = min(8, nc);
                    rc[1] = c0 + 8;
                    rn[1] = nc - rn[0];
                }
            };
            // kPreStages stages go out at once; the rest once the consumers'
            // activation loads have returned (they are not queued behind the
            // weight stream), while the consumers still stage activations.
            // From then on stages up to kPrefetchAhead ahead are prefetched
            // into L2, so a ring entry's refill reads L2 and the weight
            // stream runs through the prologue: more bytes in flight than
            // the ring holds.
            int pf = kPreStages + 1;  // next stage to prefetch
            for (int i = 0; ok && i < n_stages; ++i) {
                const int slot = i % p.S;
                // a ring entry (codes and scale scratch) is refilled once
                // every consumer warp is done with it
                bool w = i != kPreStages || mbar_wait(aload, 0);
                w = w && (i < p.S || mbar_wait(&empty[slot], ((i / p.S) - 1) & 1));
                if (!__all_sync(0xffffffffu, w)) {
                    if (lane == 0) lanes_error();
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    int rc[2], rn[2];  // first column and count of each region
                    stage_regions(i, rc, rn);
                    unsigned char *dst = smem + (size_t)slot * p.stage_bytes;
                    s_seq[slot] = i;  // published by the release of the arrive below
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(rn[0] + rn[1]) * cb);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        if (rn[r] == 0) continue;
                        const int m = NMAT == 2 ? r : 0;
                        const uint4 *src = p.Bq[m] + (size_t)rc[r] * (p.KW / 4);
                        if (!split) {
                            // whole columns: one run
                            bulk_g2s(dst + (r ? off_reg1 : 0u), src, (uint32_t)rn[r] * cb, &full[slot]);
                        } else {
                            // the chunk of each column (16-byte aligned: 64 bytes a block)
                            for (int q = 0; q < rn[r]; ++q)
                                bulk_g2s(dst + (r ? off_reg1 : 0u) + (uint32_t)q * cb,
                                         src + (size_t)q * (p.KW / 4) + (size_t)kbc0 * 4, cb, &full[slot]);
                        }
                    }
                }
                issued = i + 1;
                if (lane == 0 && i >= kPreStages) {
                    for (; pf < n_stages && pf <= i + kPrefetchAhead; ++pf) {
                        int pc[2], pn[2];
                        stage_regions(pf, pc, pn);
                        if (split) {
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int m = NMAT == 2 ? r : 0;
                                for (int q = 0; q < pn[r]; ++q)
                                    prefetch_l2(p.Bq[m] + (size_t)(pc[r] + q) * (p.KW / 4) + (size_t)kbc0 * 4, cb);
                            }
                        } else if constexpr (NMAT == 2) {
#pragma unroll
                            for (int r = 0; r < 2; ++r)
                                prefetch_l2(p.Bq[r] + (size_t)pc[r] * (p.KW / 4), (uint32_t)pn[r] * cb);
                        } else {
                            // the two regions are one contiguous run of columns
                            prefetch_l2(p.Bq[0] + (size_t)pc[0] * (p.KW / 4), (uint32_t)(pn[0] + pn[1]) * cb);
                        }
                    }
                }
            }
            if (!ok && lane == 0) {
                // leave no copy in flight into this CTA's shared memory
                for (int i = (issued > p.S ? issued - p.S : 0); i < issued; ++i)
                    (void)mbar_wait(&full[i % p.S], (i / p.S) & 1);
            }
        }
        __syncwarp();
        lanes_cluster_wait();
        return;
    }

    // =====================================================================
    // Scale warp: each stage's scale scratch, as soon as its ring entry is
    // free (the consumer warps are done with stage i - S).
    // =====================================================================
    if (warp == kScaleWarp) {
        lanes_cluster_arrive();
        lanes_bar(3, 96);  // the producer has initialised the mbarriers
        // Stage i's scale scratch: the scales, then the zeros, of this CTA's
        // groups (at most 32) for each of the 16 MMA rows, 32 floats a row;
        // the 4-group piece c of row r sits at piece c ^ (r & 7), so the 8
        // rows a load instruction reads fall in distinct banks.  Copied
        // straight from global memory by cp.async, 16 bytes (4 groups) at a
        // time where the rows allow it; each lane's copies arrive on sfull
        // when they land (32 arrivals), so no warp waits for the scales'
        // round trip under the weight stream.
        const int nch = (GL + 3) >> 2;  // 4-group pieces per row (at most 8)
        // floats per copy: 4 where every row's piece starts 16-byte aligned,
        // 2 where 8-byte, else 1
        uintptr_t align = 0;
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
            align |= reinterpret_cast<uintptr_t>(p.scales[m]) | reinterpret_cast<uintptr_t>(p.zeros[m]);
        const int vec = ((p.G | g_lo) & 3) == 0 && (align & 15u) == 0 ? 4
                        : ((p.G | g_lo) & 1) == 0 && (align & 7u) == 0 ? 2 : 1;
        auto copy_scales = [&](int i) {
            const int slot = i % p.S;
            float *scr = reinterpret_cast<float *>(smem + p.off_scr) + (size_t)slot * 32 * 32;
            const int lc0 = i * TCOLS;
            // lane: piece c = lane & 7 of MMA rows (lane >> 3) + 4 k, k = 0..3
            const int c = lane & 7;
            if (c < nch) {
                const int n = min(4, GL - 4 * c);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = (lane >> 3) + 4 * k;  // MMA row
                    int m, lc;
                    if constexpr (NMAT == 2) {
                        m = r & 1;
                        lc = lc0 + (r >> 1);
                    } else {
                        m = 0;
                        lc = lc0 + 8 * (r & 1) + (r >> 1);
                    }
                    lc = lc < ncols ? lc : 0;  // past the range: any valid row (discarded)
                    const size_t off = (size_t)(col_begin + lc) * p.G + g_lo + 4 * c;
                    float *d = scr + r * 32 + 4 * (c ^ (r & 7));
#pragma unroll
                    for (int arr = 0; arr < 2; ++arr) {  // scales, zeros
                        const float *src = (arr ? p.zeros[m] : p.scales[m]) + off;
                        float *da = d + arr * 16 * 32;
                        if (vec == 4) {
                            lanes_cp_async_16(da, src, 4u * (uint32_t)n);
                        } else if (vec == 2) {
                            lanes_cp_async_8(da, src, n >= 2 ? 8u : 4u);
                            if (n > 2) lanes_cp_async_8(da + 2, src + 2, n >= 4 ? 8u : 4u);
                        } else {
                            for (int e = 0; e < n; ++e) lanes_cp_async_4(da + e, src + e);
                        }
                    }
                }
            }
            lanes_cp_async_arrive(&sfull[slot]);
        };

        for (int i = 0; i < n_stages; ++i) {
            if (i >= p.S &&
                !__all_sync(0xffffffffu, mbar_wait(&empty[i % p.S], ((i / p.S) - 1) & 1))) {
                lanes_error();  // the consumers' scratch waits then expire as well
                break;
            }
            copy_scales(i);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");  // no copy of this warp in flight at exit
        __syncwarp();
        lanes_cluster_wait();
        return;
    }

    // =====================================================================
    // Helper warp: per stage, in order, the sum of the 16 consumer warps'
    // partials in warp order (split K: then the other ranks' sums in rank
    // order, in rank 0), the norm's inverse RMS and the outputs (its lane l
    // mirrors consumer lane l: MMA rows g and g + 8, decode lane t).  Once it
    // has read a stage's partials it releases their buffer (pfree) for the
    // consumers' partials of stage i + kPartRing.
    // =====================================================================
    if (warp == kHelperWarp) {
        lanes_cluster_arrive();
        lanes_bar(3, 96);  // the producer has initialised the mbarriers
        const int g = lane >> 2, t = lane & 3;
        const int ci = g >> 1;  // column of row g within its region (row g + 8: ci + 4)
        const bool lane_ok = t < p.M;
        const float2 *part = reinterpret_cast<const float2 *>(smem + p.off_part);  // [kPartRing][warps][32]
        // split K: rank 0's [kCombine][kMaxSplit - 1][32] partial sums of the other ranks
        const float2 *cmb = reinterpret_cast<const float2 *>(smem + p.off_cmb);
        const uint32_t cmb_r0 = split ? lanes_mapa(smem_addr(smem + p.off_cmb), 0u) : 0u;
        const uint32_t cfull_r0 = split ? lanes_mapa(smem_addr(cfull), 0u) : 0u;
        bool hfail = false;
        // the sum of stage j's partials and its outputs
        auto reduce_stage = [&](int j) {
            const int slot = j % kPartRing;
            if (!hfail && !__all_sync(0xffffffffu, mbar_wait(&pbar[slot], (j / kPartRing) & 1))) {
                lanes_error();
                hfail = true;
            }
            float a0 = 0.0f, a8 = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float2 v = part[((size_t)slot * kConsumerWarps + w) * 32 + lane];
                a0 += v.x;
                a8 += v.y;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&pfree[slot]);  // the consumers may rewrite the buffer
            if (split) {
                // the chunks' sums meet in rank 0, added in rank order
                const int cs = j % kCombine;
                const uint32_t cpar = (uint32_t)(j / kCombine) & 1u;
                if (crank != 0) {
                    // rank 0 has read entry cs's stage j - kCombine
                    if (j >= kCombine && !hfail &&
                        !__all_sync(0xffffffffu, mbar_wait(&cfree[cs], cpar ^ 1u))) {
                        lanes_error();
                        hfail = true;
                    }
                    if (hfail) a0 = a8 = __int_as_float(0x7fffffff);
                    const uint32_t o = (uint32_t)((cs * (kMaxSplit - 1) + (int)crank - 1) * 32 + lane) * 8u;
                    st_async_v2(cmb_r0 + o, __float_as_uint(a0), __float_as_uint(a8), cfull_r0 + 8u * (uint32_t)cs);
                    return;  // the outputs are rank 0's
                }
                if (lane == 0) mbar_arrive_expect_tx(&cfull[cs], (uint32_t)(p.ks - 1) * 32u * 8u);
                if (!hfail && !__all_sync(0xffffffffu, mbar_wait(&cfull[cs], cpar))) {
                    lanes_error();
                    hfail = true;
                }
                for (int r = 1; r < p.ks; ++r) {
                    const float2 v = cmb[(cs * (kMaxSplit - 1) + r - 1) * 32 + lane];
                    a0 += v.x;
                    a8 += v.y;
                }
                __syncwarp();
                // entry cs is free again on every rank
                if (lane > 0 && lane < p.ks) lanes_remote_arrive(lanes_mapa(smem_addr(&cfree[cs]), (uint32_t)lane));
            }
            if constexpr (NORM) {
                const float inv = s_inv[t];
                a0 *= inv;
                a8 *= inv;
            }
            if (hfail) a0 = a8 = __int_as_float(0x7fffffff);
            const int c0 = col_begin + j * TCOLS;
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
        };
        for (int j = 0; j < n_stages; ++j) reduce_stage(j);
        if (split && crank != 0 && !hfail) {
            // rank 0's last remote arrives have landed here before this CTA exits
            for (int j = max(0, n_stages - kCombine); j < n_stages; ++j) {
                if (!__all_sync(0xffffffffu, mbar_wait(&cfree[j % kCombine], (uint32_t)(j / kCombine) & 1u))) {
                    lanes_error();
                    break;
                }
            }
        }
        __syncwarp();
        lanes_cluster_wait();
        return;
    }

    // =====================================================================
    // Consumer warps: prologue.  One warp load instruction reads one 128-
    // activation block of one lane (lane l: activations 4l .. 4l + 3), so the
    // loads are fully coalesced.  A warp takes 4 / NP k-blocks of every lane
    // per pass (U = 4 units), all its loads issued before any is used (one
    // round trip under the weight stream); the loop bounds are uniform per
    // warp.  Per unit: the block's largest magnitude and sums are reduce-
    // scattered over the warp, the scales gathered back from the unit's owner
    // lane; X = rint(x 2^k) = 2048 h + l with l in [-1024, 1023] (both exact
    // in fp16: every MMA product and partial sum is an integer times 2^-24
    // below 2^24 of them, so a block's dot products are exact and the integer
    // part of the zero point comes off exactly through the piece sums).  Codes
    // j and j + 4 of a word (lanes 2w and 2w + 1) meet in one xor-1 shuffle
    // per piece; the odd code positions take h / 16 and l / 16 (their codes
    // are 16 q).  Stored: the pieces in the MMA's B layout [block][pair]
    // [n = 2m + part][t][8 halves], and per unit {2^(24-k), sum h 2^-24,
    // sum l 2^-24, sum x}.
    // =====================================================================
    const int ctid = threadIdx.x;
    lanes_cluster_arrive();
    lanes_dependency_wait();
    float sq[NP];
#pragma unroll
    for (int m = 0; m < NP; ++m) sq[m] = 0.0f;
    const bool cta0 = blockIdx.x == 0;
    // the first cluster writes residual_out (each CTA the blocks it stages)
    const bool cl0 = (int)blockIdx.x < (split ? p.ks : 2);
    constexpr bool TWO = PRO != kProNone;  // A_b (norm) or the gate vector
    constexpr int PB = 4 / NP;  // k-blocks per warp per pass (4 block-lane units)
    constexpr int U = PB * NP;
    const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const int par = lane & 1;  // codes 0-3 (0) or 4-7 (1) of word lane >> 1
    const int wsl = lane >> 1;
    // this lane's 8 bytes within a block's B area, lane 0 of the MMA's N
    const uint32_t act_lane = (uint32_t)(wsl & 3) * (2 * NP) * 64u + (uint32_t)(wsl >> 2) * 16u + 8u * par;
    // every consumer thread passes named barrier 4 once, before any mbarrier
    // use: the producer arrives there after initialising the mbarriers
    lanes_bar(4, kBar2Threads);
    // the cluster's mbarriers are initialised once every thread of it has
    // arrived; the partner's staging area, block factors and peerb (split K:
    // rank 0's square sums and peerb), seen from here
    lanes_cluster_wait();
    const uint32_t target = split ? 0u : peer;  // a rank of this cluster
    const uint32_t act_r = lanes_mapa(smem_addr(s_act), target);  // (pairs only)
    const uint32_t fx_r = lanes_mapa(smem_addr(smem + p.off_fx), target);
    const uint32_t sqp_r = lanes_mapa(smem_addr(s_sqp), target);
    const uint32_t peerb_r = lanes_mapa(smem_addr(peerb), target);
    if (ctid == 0) {
        // the bytes stored here by the cluster: pairs, the partner's pieces,
        // block factors and norm half sums; split K, the other ranks' square
        // sums in rank 0
        const uint32_t norm_bytes = NORM ? 4u * (uint32_t)NP : 0u;
        mbar_arrive_expect_tx(peerb, split ? (crank == 0 ? (uint32_t)(p.ks - 1) * norm_bytes : 0u)
                                           : (uint32_t)kb_peer * (uint32_t)NP * (2u * 32u * 8u + 16u) + norm_bytes);
    }
    bool pfail = false;
    bool arrived = kb_lo + PB * warp >= kb_hi;  // a warp without k-blocks signals at once
    if (arrived && lane == 0) mbar_arrive(aload);
    for (int kb0 = kb_lo + PB * warp; kb0 < kb_hi; kb0 += PB * kConsumerWarps) {
        float4 va[U], vb[U], vg[PB];
#pragma unroll
        for (int i = 0; i < PB; ++i) {
            const bool okb = kb0 + i < kb_hi;
            const size_t k0 = (size_t)(kbc0 + kb0 + i) * kBlock + 4 * lane;
#pragma unroll
            for (int m = 0; m < NP; ++m) {
                const bool on = okb && m < p.M;
                va[i * NP + m] = on ? __ldg(reinterpret_cast<const float4 *>(p.A + (size_t)m * p.K + k0)) : z4;
                if constexpr (TWO)
                    vb[i * NP + m] = (on && p.A_b != nullptr)
                                         ? __ldg(reinterpret_cast<const float4 *>(p.A_b + (size_t)m * p.K + k0))
                                         : z4;
            }
            if constexpr (NORM) vg[i] = okb ? __ldg(reinterpret_cast<const float4 *>(p.W_norm + k0)) : z4;
        }
        uint32_t mb[U];
        float smv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = u / NP, m = u % NP;
            float4 v = va[u];
            if constexpr (NORM) {
                const float4 a = vb[u];
                v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
                if (cl0 && kb0 + i < kb_hi && m < p.M && p.residual_out)
                    *reinterpret_cast<float4 *>(p.residual_out + (size_t)m * p.K +
                                                (size_t)(kbc0 + kb0 + i) * kBlock + 4 * lane) = v;
                float s2 = v.x * v.x;
                s2 = fmaf(v.y, v.y, s2); s2 = fmaf(v.z, v.z, s2); s2 = fmaf(v.w, v.w, s2);
                sq[m] += s2;
                const float4 gg = vg[i];
                v.x *= gg.x; v.y *= gg.y; v.z *= gg.z; v.w *= gg.w;
            } else if constexpr (TWO) {
                const float4 gg = vb[u];
                v.x = gate_input<PRO>(v.x, gg.x); v.y = gate_input<PRO>(v.y, gg.y);
                v.z = gate_input<PRO>(v.z, gg.z); v.w = gate_input<PRO>(v.w, gg.w);
            }
            va[u] = v;
            mb[u] = max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                        max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu));
            smv[u] = (v.x + v.y) + (v.z + v.w);
        }
        if (!arrived) {  // this warp's first activation loads have returned
            arrived = true;
            __syncwarp();
            if (lane == 0) mbar_arrive(aload);
        }
        // the scale of the lane's own unit, then of every unit from its owner
        const uint32_t mown = reduce_scatter<U>(mb, lane, OpMax());
        const float sown = reduce_scatter<U>(smv, lane, OpAdd());
        int kown;
        float fown;
        block_scale(mown, kown, fown);
        int shv[U], slv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = u / NP, m = u % NP;
            const int k = __shfl_sync(0xffffffffu, kown, rs_owner<U>(u));
            const bool bad = k == kBadScale;
            const float xv[4] = {va[u].x, va[u].y, va[u].z, va[u].w};
            int h[4], l[4];
            int sh = 0, sl = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int X = bad ? 0 : __float2int_rn(mul_pow2(xv[j], k));
                h[j] = (X + 1024) >> 11;
                l[j] = X - (h[j] << 11);
                sh += h[j];
                sl += l[j];
            }
            shv[u] = sh;
            slv[u] = sl;
            // own halves and the other lane's: (piece of code a, piece of code b / 16)
            const uint32_t hown = par ? piece_pair(h[2], h[3]) : piece_pair(h[0], h[1]);
            const uint32_t hsnd = par ? piece_pair(h[0], h[1]) : piece_pair(h[2], h[3]);
            const uint32_t lown = par ? piece_pair(l[2], l[3]) : piece_pair(l[0], l[1]);
            const uint32_t lsnd = par ? piece_pair(l[0], l[1]) : piece_pair(l[2], l[3]);
            const uint32_t hrcv = __shfl_xor_sync(0xffffffffu, hsnd, 1);
            const uint32_t lrcv = __shfl_xor_sync(0xffffffffu, lsnd, 1);
            // even lane: (code 0, code 4), (code 1, code 5); odd: (2, 6), (3, 7)
            const uint32_t ha = par ? hrcv : hown, hb = par ? hown : hrcv;
            const uint32_t la = par ? lrcv : lown, lb = par ? lown : lrcv;
            if (kb0 + i < kb_hi) {
                const uint32_t o = (uint32_t)(kb0 + i) * 4u * (2 * NP) * 64u + (uint32_t)(2 * m) * 64u + act_lane;
                const uint32_t h0 = __byte_perm(ha, hb, 0x5410), h1 = __byte_perm(ha, hb, 0x7632);
                const uint32_t l0 = __byte_perm(la, lb, 0x5410), l1 = __byte_perm(la, lb, 0x7632);
                *reinterpret_cast<uint2 *>(s_act + o) = make_uint2(h0, h1);
                *reinterpret_cast<uint2 *>(s_act + o + 64) = make_uint2(l0, l1);
                if (!split) {  // and the partner's copy
                    st_async_v2(act_r + o, h0, h1, peerb_r);
                    st_async_v2(act_r + o + 64, l0, l1, peerb_r);
                }
            }
        }
        const int shown = reduce_scatter<U>(shv, lane, OpAdd());
        const int slown = reduce_scatter<U>(slv, lane, OpAdd());
        const int uo = rs_unit<U>(lane);
        if (lane == rs_owner<U>(uo) && kb0 + uo / NP < kb_hi) {
            const float e24 = 5.9604644775390625e-8f;  // 2^-24
            const uint32_t o = ((uint32_t)(kb0 + uo / NP) * 4u + (uint32_t)(uo % NP)) * 16u;
            const float4 v = make_float4(fown, (float)shown * e24, (float)slown * e24, sown);
            *reinterpret_cast<float4 *>(smem + p.off_fx + o) = v;
            if (!split) st_async_v4(fx_r + o, v, peerb_r);
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
    }
    float own = 0.0f;  // this CTA's part of a lane's square sum (threads ctid < NP)
    if (NORM && ctid < NP) {
        for (int w = 0; w < kConsumerWarps; ++w) own += s_sq[w * 4 + ctid];
        // pairs: to the partner; split K: ranks 1.. to rank 0
        if (!split || crank != 0)
            st_async_f32(sqp_r + 4u * (uint32_t)((split ? (int)crank - 1 : 0) * 4 + ctid), own, peerb_r);
    }
    // the partner's half of the staging (and of the square sums) has landed
    if (!mbar_wait(peerb, 0)) {
        lanes_error();
        pfail = true;
    }
    if (NORM && ctid < NP) {
        if (!split) {
            // both CTAs add the halves in the same order (rank 0's first)
            const float sum = crank ? s_sqp[ctid] + own : own + s_sqp[ctid];
            s_inv[ctid] = 1.0f / sqrtf(sum / (float)p.K + p.eps);
        } else if (crank == 0) {
            // the chunks in rank order (only rank 0 applies the norm)
            float sum = own;
            for (int r = 1; r < p.ks; ++r) sum += s_sqp[(r - 1) * 4 + ctid];
            s_inv[ctid] = 1.0f / sqrtf(sum / (float)p.K + p.eps);
        }
    }
    lanes_bar(2, kBar2Threads);  // activations staged; the producer has initialised the mbarriers

    // =====================================================================
    // Consumer warps: stages.
    // =====================================================================
    // `failed` stays uniform across each warp: the MMAs need every lane
    bool failed = __any_sync(0xffffffffu, pfail);
    const int g = lane >> 2, t = lane & 3;
    // this warp's K slice: blocks [bw0, bw1)
    const int bw0 = (int)((long long)KBL * warp / kConsumerWarps);
    const int bw1 = (int)((long long)KBL * (warp + 1) / kConsumerWarps);
    float2 *part = reinterpret_cast<float2 *>(smem + p.off_part);  // [kPartRing][warps][32]
    // MMA rows g and g + 8: region g & 1, columns (g >> 1) and (g >> 1) + 4 of it
    const uint32_t row_off = ((g & 1) ? off_reg1 : 0u) + (uint32_t)(g >> 1) * cb;
    const uint32_t row8_delta = 4u * cb;
    const uint32_t b_lane_off = (uint32_t)(g * 4 + t) * 16u;
    const bool b_active = g < 2 * NP;
    // The warp's K slice is the same in every stage: its B fragments and
    // block factors stay in registers (at most kMaxWarpBlocks blocks).
    const int nb = bw1 - bw0;
    uint4 bqc[kMaxWarpBlocks][4];
    float4 fxc[kMaxWarpBlocks];
#pragma unroll
    for (int u = 0; u < kMaxWarpBlocks; ++u) {
        const int b = bw0 + (u < nb ? u : 0);
        const unsigned char *bp = s_act + (size_t)b * 4 * (2 * NP * 64) + b_lane_off;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr)
            bqc[u][pr] = (b_active && u < nb) ? *reinterpret_cast<const uint4 *>(bp + pr * (2 * NP * 64))
                                              : make_uint4(0u, 0u, 0u, 0u);
        // {2^(24-k), sum h 2^-24, sum l 2^-24, sum x} of lane t's block
        fxc[u] = u < nb ? s_fx[b * 4 + t] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }

    for (int i = 0; i < n_stages; ++i) {
        if (i == n_stages - 1 && lane == 0) lanes_dependents_launch();
        const int ring = i % p.S;
        const uint32_t ph = (uint32_t)(i / p.S) & 1u;
        if (!failed && !__all_sync(0xffffffffu, wait_shared_eq(&s_seq[ring], i) && mbar_wait(&full[ring], ph) &&
                                                    mbar_wait(&sfull[ring], ph))) {
            lanes_error();
            failed = true;
        }
        const unsigned char *st = smem + (size_t)ring * p.stage_bytes;
        // {s, z} per [group][MMA row] of this stage
        // the scales and zeros of MMA rows g and g + 8 in this stage's scratch
        // (group j at (((j >> 2) ^ g) << 2) | (j & 3) of either row)
        const float *scr = reinterpret_cast<const float *>(smem + p.off_scr) + (size_t)ring * 32 * 32;
        const float *sg0 = scr + g * 32, *sg8 = scr + (g + 8) * 32;
        const float *zg0 = scr + (16 + g) * 32, *zg8 = scr + (24 + g) * 32;

        float y0 = 0.0f, y8 = 0.0f;
        if (!failed) {
            const unsigned char *ra = st + row_off;
            // NBL (1 or 2) blocks from the warp's block U0 on: their codes
            // and scales first, then 2 NBL independent MMA chains
            auto run_blocks = [&](auto u0c, auto nbc) {
                constexpr int U0 = decltype(u0c)::value, NBL = decltype(nbc)::value;
                uint4 wa[NBL], wb[NBL];
                float2 sz0[NBL], sz8[NBL];
#pragma unroll
                for (int u = 0; u < NBL; ++u) {
                    const int b = bw0 + U0 + u;
                    wa[u] = *reinterpret_cast<const uint4 *>(ra + b * 64 + t * 16);
                    wb[u] = *reinterpret_cast<const uint4 *>(ra + row8_delta + b * 64 + t * 16);
                    const int j = b >> p.bpg_shift;
                    const int js = (((j >> 2) ^ g) << 2) | (j & 3);
                    sz0[u] = make_float2(sg0[js], zg0[js]);  // {s, z} of row g
                    sz8[u] = make_float2(sg8[js], zg8[js]);
                }
                float d1[NBL][4], d2[NBL][4];
#pragma unroll
                for (int u = 0; u < NBL; ++u)
#pragma unroll
                    for (int k = 0; k < 4; ++k) d1[u][k] = d2[u][k] = 0.0f;
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {
#pragma unroll
                    for (int u = 0; u < NBL; ++u) {
                        const uint4 bq = bqc[U0 + u][pr];
                        const uint32_t w0 = pr == 0 ? wa[u].x : pr == 1 ? wa[u].y : pr == 2 ? wa[u].z : wa[u].w;
                        const uint32_t w8 = pr == 0 ? wb[u].x : pr == 1 ? wb[u].y : pr == 2 ? wb[u].z : wb[u].w;
                        mma_f16(d1[u], w0 & 0x000F000Fu, w8 & 0x000F000Fu, w0 & 0x00F000F0u, w8 & 0x00F000F0u,
                                bq.x, bq.y);
                        const uint32_t v0 = w0 >> 8, v8 = w8 >> 8;
                        mma_f16(d2[u], v0 & 0x000F000Fu, v8 & 0x000F000Fu, v0 & 0x00F000F0u, v8 & 0x00F000F0u,
                                bq.z, bq.w);
                    }
                }
#pragma unroll
                for (int u = 0; u < NBL; ++u) {
                    const float4 fx = fxc[U0 + u];
                    // zi: the zero's integer part (clamped to the code range)
                    const float zi0 = rintf(fminf(fmaxf(sz0[u].y, 0.0f), 15.0f));
                    const float zi8 = rintf(fminf(fmaxf(sz8[u].y, 0.0f), 15.0f));
                    // exact: sum (q - zi) h and sum (q - zi) l, times 2^-24
                    const float h0 = fmaf(-zi0, fx.y, d1[u][0] + d2[u][0]);
                    const float l0 = fmaf(-zi0, fx.z, d1[u][1] + d2[u][1]);
                    const float h8 = fmaf(-zi8, fx.y, d1[u][2] + d2[u][2]);
                    const float l8 = fmaf(-zi8, fx.z, d1[u][3] + d2[u][3]);
                    // y += s * (sum (q - zi) x - (z - zi) X)
                    y0 = fmaf(sz0[u].x, fmaf(zi0 - sz0[u].y, fx.w, fmaf(h0, 2048.0f, l0) * fx.x), y0);
                    y8 = fmaf(sz8[u].x, fmaf(zi8 - sz8[u].y, fx.w, fmaf(h8, 2048.0f, l8) * fx.x), y8);
                }
            };
            // the warp's blocks two at a time, an odd last one alone (nb is
            // uniform across the warp)
            static_assert(kMaxWarpBlocks <= 3, "blocks per warp");
            if (nb >= 2) run_blocks(IntC<0>{}, IntC<2>{});
            else if (nb == 1) run_blocks(IntC<0>{}, IntC<1>{});
            if (nb == 3) run_blocks(IntC<2>{}, IntC<1>{});
        }

        // this warp is done with the stage's codes and scratch
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[ring]);
        // its partial sums go to the helper warp (partial buffer i mod
        // kPartRing, once the helper has read stage i - kPartRing's)
        const int pr_slot = i % kPartRing;
        if (i >= kPartRing && !failed &&
            !__all_sync(0xffffffffu, mbar_wait(&pfree[pr_slot], (uint32_t)((i / kPartRing) - 1) & 1u))) {
            lanes_error();
            failed = true;
        }
        if (failed) y0 = y8 = __int_as_float(0x7fffffff);
        part[((size_t)pr_slot * kConsumerWarps + warp) * 32 + lane] = make_float2(y0, y8);
        __syncwarp();
        if (lane == 0) mbar_arrive(&pbar[pr_slot]);
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

template <int NMAT, int PRO, int EPI, int NP, bool SPLIT>
cudaError_t launch_lanes_variant(const LanesParams &prm, size_t smem, cudaStream_t stream)
{
    auto kern = lanes_matvec_kernel<NMAT, PRO, EPI, NP, SPLIT>;
    int dev = 0, sms = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    constexpr int kMaxDevices = 64;
    static std::atomic<unsigned char> smem_ready[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices || !smem_ready[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   (int)cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < kMaxDevices) smem_ready[dev].store(1, std::memory_order_release);
    }
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    // Clusters of 2 (pairs sharing the activation staging) or of ks (split
    // K): as many as are resident, no more than the columns need (a CTA may
    // get none)
    const int cd = prm.ks > 1 ? prm.ks : 2;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cd;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int clusters = sms / cd;
    cfg.gridDim = dim3((unsigned)(cd * clusters));
    int resident = 0;
    if (cudaOccupancyMaxActiveClusters(&resident, kern, &cfg) == cudaSuccess && resident > 0 &&
        resident < clusters)
        clusters = resident;
    const int need = prm.ks > 1 ? prm.n_units : (prm.n_units + 1) / 2;
    if (clusters > need) clusters = need;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3((unsigned)(cd * clusters));
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int NMAT, int PRO, int EPI>
cudaError_t launch_lanes_np(const LanesParams &prm, size_t smem, cudaStream_t stream)
{
    if (prm.ks > 1)
        return prm.M <= 2 ? launch_lanes_variant<NMAT, PRO, EPI, 2, true>(prm, smem, stream)
                          : launch_lanes_variant<NMAT, PRO, EPI, 4, true>(prm, smem, stream);
    return prm.M <= 2 ? launch_lanes_variant<NMAT, PRO, EPI, 2, false>(prm, smem, stream)
                      : launch_lanes_variant<NMAT, PRO, EPI, 4, false>(prm, smem, stream);
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
    prm.bpg = call.gs / kBlock;
    if ((prm.bpg & (prm.bpg - 1)) != 0) return false;  // group of a block by a shift
    prm.bpg_shift = 0;
    while ((1 << prm.bpg_shift) < prm.bpg) ++prm.bpg_shift;
    // A CTA's chunk of K: at most 32 scale groups (the helper holds a
    // stage's scales as one group per lane) and at most kMaxWarpBlocks blocks
    // per consumer warp (its activations stay in registers).  All of K in
    // one CTA (pairs) where it fits; else the fewest chunks per cluster that
    // give each warp at most kSplitWarpBlocks blocks (at most kMaxWarpBlocks).
    auto largest_chunk = [&](int ks) {  // groups
        int most = 0;
        for (int r = 0; r < ks; ++r)
            most = max(most, chunk_group(prm.G, ks, r + 1) - chunk_group(prm.G, ks, r));
        return most;
    };
    auto chunk_fits = [&](int ks, int warp_blocks) {
        // every chunk holds at least one group (aligned bounds can merge
        // neighbours when G is small): no empty copies, no idle rank
        for (int r = 0; r < ks; ++r)
            if (chunk_group(prm.G, ks, r + 1) <= chunk_group(prm.G, ks, r)) return false;
        const int gmax = largest_chunk(ks);
        return gmax <= 32 && (gmax * prm.bpg + kConsumerWarps - 1) / kConsumerWarps <= warp_blocks;
    };
    // clusters of 2 or 4 before 3 (3-CTA clusters measured slower: they pack
    // fewer SMs per GPC)
    constexpr int kSplitOrder[3] = {2, 4, 3};
    int ks = 0;
    if (chunk_fits(1, kMaxWarpBlocks)) {
        ks = 1;
    } else {
        for (int o = 0; o < 3 && ks == 0; ++o)
            if (kSplitOrder[o] <= kMaxSplit && chunk_fits(kSplitOrder[o], kSplitWarpBlocks)) ks = kSplitOrder[o];
        for (int o = 0; o < 3 && ks == 0; ++o)
            if (kSplitOrder[o] <= kMaxSplit && chunk_fits(kSplitOrder[o], kMaxWarpBlocks)) ks = kSplitOrder[o];
        if (ks == 0) return false;
    }
    prm.ks = ks;
    prm.Gs = largest_chunk(ks);
    const int KBC = prm.Gs * prm.bpg;  // the largest chunk's blocks
    prm.unit = 1;
    prm.n_units = call.N;
    const int NP = call.M <= 2 ? 2 : 4;
    const uint32_t reg_bytes = 8u * (uint32_t)KBC * 64u;  // a multiple of 512
    const uint32_t stage = round_up(reg_bytes + 64u + reg_bytes, 128u);
    const uint32_t act_bytes = (uint32_t)KBC * 4u * (uint32_t)(2 * NP) * 64u;
    const uint32_t fx_bytes = (uint32_t)KBC * 4u * 16u;
    const uint32_t misc_bytes = 384u;  // inverse RMS [4], square sums [warps][4], the others' [3][4]
    const uint32_t cmb_bytes = ks > 1 ? (uint32_t)kCombine * (kMaxSplit - 1) * 32u * 8u : 0u;
    const uint32_t bar_bytes = (5 * kMaxStages + 2 + 2 * kCombine) * 8u + kMaxStages * 4u;
    // per ring entry: the codes and the scale scratch
    const uint32_t scr_per_stage = 32u * 32u * 4u;  // 16 rows of scales, 16 of zeros, 32 groups each
    const uint32_t part_bytes = (uint32_t)kPartRing * kConsumerWarps * 32u * 8u;  // the partial ring
    const uint32_t per_stage = stage + scr_per_stage;
    const uint32_t fixed = act_bytes + fx_bytes + part_bytes + misc_bytes + cmb_bytes + bar_bytes + 4u * 128u;
    if (fixed + 2u * per_stage > kSmemLimit) return false;
    int S = (int)((kSmemLimit - fixed) / per_stage);
    if (S > kMaxStages) S = kMaxStages;
    prm.S = S;
    prm.stage_bytes = stage;
    uint32_t off = round_up((uint32_t)S * stage, 128u);
    prm.off_act = off;
    off += act_bytes;
    prm.off_fx = off;
    off += round_up(fx_bytes, 128u);
    prm.off_part = off;
    off += round_up(part_bytes, 128u);
    prm.off_scr = off;
    off += round_up((uint32_t)S * scr_per_stage, 128u);
    prm.off_misc = off;
    off += misc_bytes;
    prm.off_cmb = off;
    off += round_up(cmb_bytes, 128u);
    prm.off_bar = off;
    off += bar_bytes;
    smem = off;
    return smem <= kSmemLimit;
}

}  // namespace

bool lanes_path_supported(const Call &call)
{
    if (call.M < 2 || call.M > 4) return false;
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

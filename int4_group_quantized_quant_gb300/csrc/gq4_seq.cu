// gq4_seq.cu -- one persistent launch for a sequence of one-lane (M = 1)
// calls: plain, quad routing, RMSNorm prologue and SiLU-gated gate/up, in
// order, each call free to read what the earlier ones wrote.
//
// Operation of each call: the same as the single-call kernels
// (gerbil moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 / WGSL_NORM_MATVEC_INT4;
// the executor runs a decode step as such a list of dispatches).
//
// Why one launch: a one-lane call streams a few MB; per call, a separate
// launch pays the launch gap, an activation prologue during which the weight
// ring is nearly empty, the ring fill and the tail of the slowest warp.  Here
// one CTA per SM (all resident: cooperative launch) keeps a single weight
// ring across calls:
//   * The producer warp streams the stages of call i+1 into the ring as soon
//     as slots free up, i.e. during the tail of call i and during call i+1's
//     activation prologue, so that prologue runs with the ring already full
//     and no weight traffic competing with its activation loads.
//   * A stage holds whole columns of one call: their packed codes and their
//     scale and zero rows (so no per-call row buffer has to be swapped).
//   * Consumers finish call i, then meet at a grid barrier (one growing
//     atomic counter in a caller-provided workspace; waits bounded in time)
//     before staging call i+1's activations, which may be call i's outputs.  Activations are read through L2 (ld.global.cg),
//     never from a possibly stale L1 line.
//   * Within a call the arithmetic is the one-lane streaming kernel's
//     (gq4_onelane.cuh): the activations staged once per CTA as 24-bit
//     fixed-point byte pieces with a power-of-two scale per chunk group;
//     warp slots of four columns (or two gate and two up columns); integer
//     dp4a sums per chunk group with the zero's integer part taken out
//     exactly and its fractional part applied through the group's
//     activation sum; one xor reduce-scatter per slot.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gq4_device.cuh"
#include "gq4_internal.h"
#include "gq4_onelane.cuh"
#include "gq4_tma.cuh"

namespace gq4 {

// Sticky device-side error word of this path (bit 2: a wait timed out).
__device__ unsigned int g_seq_error = 0;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kActBatch = 4;  // activation float4 per consumer thread per prologue batch (register budget: the kernel holds every call variant)
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kCT = kConsumerWarps * 32;
constexpr int kSPW = 4;          // weight streams per warp slot
constexpr int kMaxStages = 16;
constexpr int kMaxCalls = kSeqMaxCalls;  // calls per launch (kernel-parameter space)
constexpr uint32_t kSmemLimit = 220u * 1024u;
constexpr uint32_t kStageMin = 16u * 1024u;

// Consumer code of a call: (matrices, norm prologue, epilogue) x R.
enum Variant : int {
    kVarStore = 0,      // one matrix, store
    kVarNormStore = 1,  // one matrix, norm prologue, store
    kVarQuad = 2,       // one matrix, quad routing
    kVarGated = 3,      // gate/up, SiLU-gated
    kVarNormGated = 4,  // gate/up, norm prologue, SiLU-gated
};

// One call as the kernel sees it (planned on the host).
struct SeqCall {
    int variant;       // Variant
    int R;             // 32-code chunks per chunk group (1 or 2)
    int nmat;
    int K, N, KC, G, KP;
    int unit;          // column granularity: scale rows of a unit start 16-byte aligned
    int n_units;
    int cps;           // columns per warp slot (per matrix)
    int wps;           // warp slots per stage
    int stage_cols;    // wps * cps
    uint32_t mat_w;    // bytes of packed codes per matrix in a stage (stage_cols * KC * 16)
    uint32_t mat_sz;   // bytes of one row array per matrix in a stage (16-byte multiple)
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

struct SeqParams {
    int n_calls;
    int S;                    // ring depth
    uint32_t stage_bytes;
    uint32_t off_act, off_norm, off_bar;
    uint32_t magic_bits;      // 0x0F0F0F0F (even-code mask), read from the parameter bank
    unsigned int *bar_count;  // grid barrier: arrivals so far in this launch
    unsigned int *bar_exit;   // CTAs that have finished this launch
    SeqCall calls[kMaxCalls];
};
static_assert(sizeof(SeqParams) <= 32000, "kernel parameters");

__device__ __forceinline__ void named_barrier_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void seq_error()
{
    atomicOr(&g_seq_error, 4u);
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned int atom_add_release_gpu(unsigned int *p, unsigned int v)
{
    unsigned int old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed_gpu(unsigned int *p, unsigned int v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier among the consumer threads of every CTA (thread `ctid`
// 0 of each CTA does the global part).  One counter grows through the
// launch: every CTA adds 1 per boundary with release semantics (its outputs,
// ordered before thread 0 by the CTA barrier, are published by it), and
// waits, bounded in time, to acquire a count of at least `target`, the next
// multiple of the grid size.  One release per CTA and no reset between
// boundaries keep a single gpu-scope release -- microseconds under the
// weight stream's traffic -- on the critical path.  Returns false on expiry.
__device__ bool grid_barrier(const SeqParams &p, int ctid, unsigned int &target)
{
    bool ok = true;
    named_barrier_sync(1, kCT);  // every output of this CTA's call is written
    if (ctid == 0) {
        target += gridDim.x;
        (void)atom_add_release_gpu(p.bar_count, 1u);
        const unsigned long long t0 = global_timer_ns();
        while ((int)(ld_acquire_gpu(p.bar_count) - target) < 0) {
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                seq_error();
                ok = false;
                break;
            }
            __nanosleep(32);
        }
    }
    named_barrier_sync(1, kCT);
    return ok;
}

// This CTA's contiguous column range of a call, in whole units.
__device__ __forceinline__ void cta_columns(const SeqCall &c, int &col_begin, int &col_end)
{
    const int u0 = (int)((long long)c.n_units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)c.n_units * (blockIdx.x + 1) / gridDim.x);
    col_begin = u0 * c.unit;
    col_end = min(u1 * c.unit, c.N);
    if (col_end < col_begin) col_end = col_begin;
}

__device__ __forceinline__ int stages_of(const SeqCall &c, int ncols)
{
    return (ncols + c.stage_cols - 1) / c.stage_cols;
}


// Shared-memory objects of the kernel.
struct SeqShared {
    uint64_t *full, *empty, *ready;
    int *s_seq;    // stage number a ring entry holds (guards against parity ABA)
    int *s_done;   // warp slots of the ring entry finished so far
};

// Consumer warps: one call.  Stages its activations, then takes warp slots
// round-robin from the ring entries gstage0, gstage0 + 1, ... of this call.
template <int NMAT, bool NORM, int EPI, int R>
__device__ __forceinline__ void consume_call(const SeqParams &p, const SeqCall &c, unsigned char *smem,
                                             const SeqShared &sh, bool first_call, int gstage0,
                                             bool &failed)
{
    constexpr int CPS = NMAT == 2 ? kSPW / 2 : kSPW;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ctid = threadIdx.x;
    uint4 *s_act = reinterpret_cast<uint4 *>(smem + p.off_act);
    float *s_norm = reinterpret_cast<float *>(smem + p.off_norm);
    int col_begin, col_end;
    cta_columns(c, col_begin, col_end);
    const int ncols = col_end - col_begin;
    const int n_slots = (ncols + CPS - 1) / CPS;

    // ---- prologue: activations (through L2: earlier calls may have written
    // them) ----
    // inv: the norm prologue's inverse RMS, applied to each finished dot product
    const float inv = stage_activations_i8<R, NORM ? kProNorm : kProNone, kCT, kActBatch, LoadL2>(
        c.K, c.A, c.A_b, c.W_norm, c.eps, c.residual_out, blockIdx.x == 0, s_act, s_norm, ctid, 1);
    if (first_call && ctid == 0) mbar_arrive(sh.ready);

    // ---- warp slots ----
    const uint32_t mask = p.magic_bits;
    const int swap = chunk_swap<R>(lane);
    for (int i = warp; i < n_slots; i += kConsumerWarps) {
        const int stage = i / c.wps;
        const int sub = i - stage * c.wps;
        const int g = gstage0 + stage;
        const int ring = g % p.S;
        const int lc0 = i * CPS;  // CTA-relative first column of the slot
        const int nc = min(CPS, ncols - lc0);
        if (!failed &&
            !(wait_shared_eq(&sh.s_seq[ring], g) && mbar_wait(&sh.full[ring], (g / p.S) & 1))) {
            seq_error();
            failed = true;
        }
        const unsigned char *sl = smem + (size_t)ring * p.stage_bytes;
        const int sc0 = sub * CPS;  // stage-relative first column of the slot
        const float *srow[NMAT];
        const float *zrow[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            srow[m] = reinterpret_cast<const float *>(sl + NMAT * c.mat_w + m * c.mat_sz);
            zrow[m] = reinterpret_cast<const float *>(sl + NMAT * c.mat_w + (NMAT + m) * c.mat_sz);
        }

        float acc[kSPW];
#pragma unroll
        for (int q = 0; q < kSPW; ++q) acc[q] = 0.0f;

        // The slot's packed words of stream q (a short last slot repeats its
        // column 0, whose result is then discarded).
        auto slot_words = [&](int q) -> const uint4 * {
            const int mat = NMAT == 2 ? (q / CPS) : 0;
            int lc = NMAT == 2 ? (q % CPS) : q;
            lc = lc < nc ? lc : 0;
            return reinterpret_cast<const uint4 *>(sl + mat * c.mat_w) + (size_t)(sc0 + lc) * c.KC;
        };
        // One chunk group (R chunks) of all kSPW streams.
        auto group_dot = [&](int jg, const uint4 (&wq)[kSPW][R]) {
            const int grp = chunk_group(jg * R, c.group_magic);
            float sc[kSPW], zz[kSPW];
#pragma unroll
            for (int q = 0; q < kSPW; ++q) {
                const int mat = NMAT == 2 ? (q / CPS) : 0;
                int lc = NMAT == 2 ? (q % CPS) : q;
                lc = lc < nc ? lc : 0;
                const int si = (sc0 + lc) * c.G + grp;
                sc[q] = srow[mat][si];
                zz[q] = zrow[mat][si];
            }
            chunk_group_dot_i8<kSPW, R>(s_act, jg, swap, wq, sc, zz, mask, acc);
        };

        if (!failed) {
            for (int jg = lane; jg < c.KP; jg += 32) {
                uint4 wq[kSPW][R];
#pragma unroll
                for (int q = 0; q < kSPW; ++q) {
                    const uint4 *w = slot_words(q);
#pragma unroll
                    for (int r = 0; r < R; ++r) wq[q][r] = w[jg * R + (r ^ swap)];
                }
                group_dot(jg, wq);
            }
        }
        // this warp's slot of the ring entry has been read; the last of the
        // entry's slots to finish releases it to the producer
        __syncwarp();
        if (lane == 0) {
            const int st_cols = min(c.stage_cols, ncols - stage * c.stage_cols);
            const int slots_here = (st_cols + CPS - 1) / CPS;
            if (atomicAdd(&sh.s_done[ring], 1) == slots_here - 1) {
                sh.s_done[ring] = 0;
                mbar_arrive(&sh.empty[ring]);
            }
        }

        // ---- reduce-scatter of the four streams across the warp ----
        // step 16: lanes < 16 keep streams 0,1; lanes >= 16 keep streams 2,3
        const bool hi16 = (lane & 16) != 0;
        float k0 = hi16 ? acc[2] : acc[0];
        float k1 = hi16 ? acc[3] : acc[1];
        const float s0 = hi16 ? acc[0] : acc[2];
        const float s1 = hi16 ? acc[1] : acc[3];
        k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
        k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
        // step 8: lanes with bit 3 clear keep the first, others the second
        const bool hi8 = (lane & 8) != 0;
        float total = hi8 ? k1 : k0;
        total += __shfl_xor_sync(0xffffffffu, hi8 ? k0 : k1, 8);
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
        // lane 0 -> stream 0, lane 8 -> 1, lane 16 -> 2, lane 24 -> 3
        const int q_of_lane = ((lane >> 4) << 1) | ((lane >> 3) & 1);
        if constexpr (NORM) total *= inv;
        if (failed) total = __int_as_float(0x7fffffff);

        // ---- epilogue ----
        const int c0 = col_begin + lc0;
        if constexpr (EPI == kEpiGated) {
            // streams 0, 1 are gate columns, 2, 3 the matching up columns
            const float u = __shfl_down_sync(0xffffffffu, total, 16);
            if ((lane & 7) == 0 && lane < 16) {
                const int lc = q_of_lane;
                if (lc < nc) {
                    const float gv = total;
                    c.out[0][c0 + lc] = gv / (1.0f + expf(-gv)) * u;
                }
            }
        } else {
            if ((lane & 7) == 0) {
                const int lc = q_of_lane;
                if (lc < nc) {
                    const int col = c0 + lc;
                    if constexpr (EPI == kEpiQuad) {
                        const int seg = col < c.seg_start[1] ? 0 : col < c.seg_start[2] ? 1
                                      : col < c.seg_start[3] ? 2 : 3;
                        c.out[seg][col - c.seg_start[seg]] = total;
                    } else {
                        c.out[0][col] = total;
                    }
                }
            }
        }
    }
    if constexpr (NORM) {
        if (blockIdx.x == 0 && c.norm_out)
            write_norm_out<kCT, LoadL2>(c.K, c.A, c.A_b, c.W_norm, inv, c.norm_out, ctid);
    }
}

__global__ void __launch_bounds__(kThreads, 1) seq_kernel(const __grid_constant__ SeqParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + kMaxStages;
    uint64_t *ready = empty + kMaxStages;  // consumers' first prologue done
    int *s_seq = reinterpret_cast<int *>(ready + 1);
    int *s_done = s_seq + kMaxStages;
    const SeqShared sh{full, empty, ready, s_seq, s_done};
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);  // the last warp slot of the entry to finish
            s_seq[s] = -1;
            s_done[s] = 0;
        }
        mbar_init(ready, 1);
        mbar_fence_init();
    }
    __syncthreads();

    // =====================================================================
    // Producer warp: every call's stages through one ring.
    // =====================================================================
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            int g = 0;  // ring entries issued so far (over all calls)
            bool ok = true;
            for (int ci = 0; ok && ci < p.n_calls; ++ci) {
                const SeqCall &c = p.calls[ci];
                int col_begin, col_end;
                cta_columns(c, col_begin, col_end);
                const int n_st = stages_of(c, col_end - col_begin);
                for (int i = 0; i < n_st; ++i, ++g) {
                    const int slot = g % p.S;
                    // two entries go out at once; the rest wait for the
                    // consumers' first prologue, so its activation loads are
                    // not queued behind every CTA's whole ring of weight copies
                    if (g == 2 && !mbar_wait(ready, 0)) {
                        seq_error();
                        ok = false;
                        break;
                    }
                    if (g >= p.S && !mbar_wait(&empty[slot], ((g / p.S) - 1) & 1)) {
                        seq_error();
                        ok = false;
                        break;
                    }
                    const int c0 = col_begin + i * c.stage_cols;
                    const int nc = min(c.stage_cols, col_end - c0);
                    unsigned char *dst = smem + (size_t)slot * p.stage_bytes;
                    const uint32_t w_bytes = (uint32_t)nc * (uint32_t)c.KC * 16u;
                    const uint32_t r_all = (uint32_t)nc * (uint32_t)c.G * 4u;
                    const uint32_t r_bulk = r_all & ~15u;
                    // ragged tail of the rows (only at the end of the matrix)
                    for (uint32_t b = r_bulk; b < r_all; b += 4) {
                        for (int m = 0; m < c.nmat; ++m) {
                            const size_t e = (size_t)c0 * c.G + b / 4;
                            *reinterpret_cast<float *>(dst + c.nmat * c.mat_w + m * c.mat_sz + b) =
                                c.scales[m][e];
                            *reinterpret_cast<float *>(dst + c.nmat * c.mat_w + (c.nmat + m) * c.mat_sz + b) =
                                c.zeros[m][e];
                        }
                    }
                    s_seq[slot] = g;  // published by the release of the arrive below
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)c.nmat * (w_bytes + 2u * r_bulk));
                    for (int m = 0; m < c.nmat; ++m) {
                        bulk_g2s(dst + m * c.mat_w, c.Bq[m] + (size_t)c0 * c.KC, w_bytes, &full[slot]);
                        if (r_bulk) {
                            bulk_g2s(dst + c.nmat * c.mat_w + m * c.mat_sz, c.scales[m] + (size_t)c0 * c.G,
                                     r_bulk, &full[slot]);
                            bulk_g2s(dst + c.nmat * c.mat_w + (c.nmat + m) * c.mat_sz,
                                     c.zeros[m] + (size_t)c0 * c.G, r_bulk, &full[slot]);
                        }
                    }
                }
            }
            if (!ok) {
                // leave no copy in flight into this CTA's shared memory
                for (int i = (g > p.S ? g - p.S : 0); i < g; ++i)
                    (void)mbar_wait(&full[i % p.S], (i / p.S) & 1);
            }
        }
        return;
    }

    // =====================================================================
    // Consumer warps: the calls in order, a grid barrier between calls.
    // =====================================================================
    bool failed = false;
    unsigned int target = 0;  // the barrier counter starts every launch at zero
    int g0 = 0;  // first ring entry of the current call
    for (int ci = 0; ci < p.n_calls; ++ci) {
        const SeqCall &c = p.calls[ci];
        if (ci > 0) (void)grid_barrier(p, threadIdx.x, target);
        const bool first = ci == 0;
        switch (c.variant * 2 + (c.R == 2 ? 1 : 0)) {
        case kVarStore * 2: consume_call<1, false, kEpiStore, 1>(p, c, smem, sh, first, g0, failed); break;
        case kVarStore * 2 + 1: consume_call<1, false, kEpiStore, 2>(p, c, smem, sh, first, g0, failed); break;
        case kVarNormStore * 2: consume_call<1, true, kEpiStore, 1>(p, c, smem, sh, first, g0, failed); break;
        case kVarNormStore * 2 + 1: consume_call<1, true, kEpiStore, 2>(p, c, smem, sh, first, g0, failed); break;
        case kVarQuad * 2: consume_call<1, false, kEpiQuad, 1>(p, c, smem, sh, first, g0, failed); break;
        case kVarQuad * 2 + 1: consume_call<1, false, kEpiQuad, 2>(p, c, smem, sh, first, g0, failed); break;
        case kVarGated * 2: consume_call<2, false, kEpiGated, 1>(p, c, smem, sh, first, g0, failed); break;
        case kVarGated * 2 + 1: consume_call<2, false, kEpiGated, 2>(p, c, smem, sh, first, g0, failed); break;
        case kVarNormGated * 2: consume_call<2, true, kEpiGated, 1>(p, c, smem, sh, first, g0, failed); break;
        default: consume_call<2, true, kEpiGated, 2>(p, c, smem, sh, first, g0, failed); break;
        }
        int col_begin, col_end;
        cta_columns(c, col_begin, col_end);
        g0 += stages_of(c, col_end - col_begin);
    }
    // The last CTA to finish puts both counters back to zero for the next
    // launch (which starts only after this one has ended); every CTA has
    // finished its last barrier wait before it counts itself out here.
    if (threadIdx.x == 0 && atomicAdd(p.bar_exit, 1u) == gridDim.x - 1) {
        st_relaxed_gpu(p.bar_count, 0u);
        st_relaxed_gpu(p.bar_exit, 0u);
    }
}
}  // namespace
}  // namespace gq4

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace gq4 {
namespace {

uint32_t rup(uint32_t x, uint32_t a)
{
    return (x + a - 1) / a * a;
}

int gcd_i(int a, int b)
{
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Bytes of one ring entry holding `wps` warp slots of call c.
uint32_t entry_bytes(const SeqCall &c, int wps)
{
    const uint32_t cols = (uint32_t)(wps * c.cps);
    return (uint32_t)c.nmat * (cols * (uint32_t)c.KC * 16u + 2u * rup(cols * (uint32_t)c.G * 4u, 16u));
}

// Warp slots per entry must make the entry's columns a multiple of the unit.
int slot_step(const SeqCall &c)
{
    const int l = c.cps / gcd_i(c.cps, c.unit) * c.unit;  // lcm(cps, unit)
    return l / c.cps;
}

// Shape part of a call's plan (everything but the ring geometry).
void plan_call_shape(const Call &call, SeqCall &sc)
{
    std::memset(&sc, 0, sizeof(sc));
    sc.nmat = call.nmat;
    if (call.epi == kEpiGated)
        sc.variant = call.norm ? kVarNormGated : kVarGated;
    else if (call.epi == kEpiQuad)
        sc.variant = kVarQuad;
    else
        sc.variant = call.norm ? kVarNormStore : kVarStore;
    sc.K = call.K;
    sc.N = call.N;
    sc.KC = call.K / 32;
    sc.G = call.K / call.gs;
    sc.R = (call.gs >= 64 && sc.KC % 2 == 0) ? 2 : 1;
    sc.KP = sc.KC / sc.R;
    sc.unit = 4 / gcd_i(sc.G, 4);
    sc.n_units = (call.N + sc.unit - 1) / sc.unit;
    sc.cps = call.nmat == 2 ? kSPW / 2 : kSPW;
    const unsigned long long cpg = (unsigned long long)(call.gs / 32);
    sc.group_magic = ((1ull << 40) + cpg - 1) / cpg;
    sc.A = call.A;
    if (call.norm) {
        sc.A_b = call.norm->A_b;
        sc.W_norm = call.norm->W_norm;
        sc.eps = call.norm->eps;
        sc.residual_out = call.norm->residual_out;
        sc.norm_out = call.norm->norm_out;
    }
    for (int m = 0; m < 2; ++m) {
        const int src = m < call.nmat ? m : 0;
        sc.Bq[m] = reinterpret_cast<const uint4 *>(call.Bq[src]);
        sc.scales[m] = call.scales[src];
        sc.zeros[m] = call.zeros[src];
    }
    for (int i = 0; i < 4; ++i) {
        sc.out[i] = call.out[i];
        sc.seg_start[i] = call.seg_start[i];
        sc.seg_len[i] = call.seg_len[i];
    }
}

// Ring geometry shared by the calls calls[0..n): one entry size for all.
bool plan_sequence(const Call *calls, int n, SeqParams &prm, size_t &smem)
{
    std::memset(&prm, 0, sizeof(SeqParams) - sizeof(prm.calls));
    prm.n_calls = n;
    // one entry size for the whole sequence: the largest one-slot entry of
    // any call (at least kStageMin), so that long columns (one slot per
    // entry) get as many entries in flight as shared memory allows
    uint32_t sb = kStageMin;
    int kc_max = 0;
    for (int i = 0; i < n; ++i) {
        SeqCall &sc = prm.calls[i];
        plan_call_shape(calls[i], sc);
        const uint32_t one = entry_bytes(sc, slot_step(sc));
        sb = one > sb ? one : sb;
        kc_max = sc.KC > kc_max ? sc.KC : kc_max;
    }
    sb = rup(sb, 128u);
    for (int i = 0; i < n; ++i) {
        SeqCall &sc = prm.calls[i];
        const int q = slot_step(sc);
        int wps = q;
        while (entry_bytes(sc, wps + q) <= sb) wps += q;
        sc.wps = wps;
        sc.stage_cols = wps * sc.cps;
        sc.mat_w = (uint32_t)sc.stage_cols * (uint32_t)sc.KC * 16u;
        sc.mat_sz = rup((uint32_t)sc.stage_cols * (uint32_t)sc.G * 4u, 16u);
    }
    const uint32_t act = rup((uint32_t)kc_max * 128u, 128u);
    const uint32_t bars = rup((2 * kMaxStages + 1) * 8u + 2 * kMaxStages * 4u, 128u);
    const uint32_t fixed = act + 128u + bars;
    if (fixed + 2u * sb > kSmemLimit) return false;
    int S = (int)((kSmemLimit - fixed) / sb);
    if (S > kMaxStages) S = kMaxStages;
    prm.S = S;
    prm.stage_bytes = sb;
    prm.off_act = rup((uint32_t)S * sb, 128u);
    prm.off_norm = prm.off_act + act;
    prm.off_bar = prm.off_norm + 128u;
    prm.magic_bits = 0x0F0F0F0Fu;
    smem = prm.off_bar + bars;
    return true;
}

constexpr int kMaxDevices = 64;

}  // namespace

bool sequence_plannable(const Call *calls, int n)
{
    static thread_local SeqParams prm;
    for (int i = 0; i < n; ++i)
        if (calls[i].M != 1) return false;
    // one CTA of the kernel must fit on every SM (cooperative launch)
    int dev = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaFuncSetAttribute(seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit) !=
        cudaSuccess)
        return false;
    size_t smem = 0;
    for (int i0 = 0; i0 < n; i0 += kMaxCalls) {
        const int m = n - i0 < kMaxCalls ? n - i0 : kMaxCalls;
        if (!plan_sequence(calls + i0, m, prm, smem)) return false;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, seq_kernel, kThreads, smem) != cudaSuccess ||
            per_sm < 1)
            return false;
    }
    return true;
}

cudaError_t launch_sequence(const Call *calls, int n, void *workspace, cudaStream_t stream)
{
    static thread_local SeqParams prm;
    int dev = 0, sms = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    static std::atomic<unsigned char> ready[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices || !ready[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < kMaxDevices) ready[dev].store(1, std::memory_order_release);
    }
    for (int i0 = 0; i0 < n; i0 += kMaxCalls) {
        const int m = n - i0 < kMaxCalls ? n - i0 : kMaxCalls;
        size_t smem = 0;
        if (!plan_sequence(calls + i0, m, prm, smem)) return cudaErrorInvalidValue;
        prm.bar_count = reinterpret_cast<unsigned int *>(workspace);
        prm.bar_exit = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(workspace) + 64);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3((unsigned)sms);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((err = cudaLaunchKernelEx(&cfg, seq_kernel, prm)) != cudaSuccess) return err;
    }
    return cudaGetLastError();
}

// Scratch of the allocation-free sequence entry point: the grid barrier's
// counters in a fixed device array of this library instead of a caller
// buffer (zero when the module loads; a completed launch leaves it zero).
constexpr size_t kSeqStaticScratchBytes = 256;
static_assert(kSeqWorkspaceBytes <= kSeqStaticScratchBytes, "sequence scratch exceeds its static array");
__device__ __align__(256) unsigned char g_seq_static_scratch[kSeqStaticScratchBytes];

size_t seq_static_scratch_bytes()
{
    return kSeqStaticScratchBytes;
}

cudaError_t seq_static_scratch(void **ptr)
{
    // Looked up once per device, with that device current (the caller's).
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_seq_static_scratch);
        if (err != cudaSuccess) return err;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

cudaError_t read_seq_device_error(unsigned int *bits, bool clear)
{
    cudaError_t err = cudaMemcpyFromSymbol(bits, g_seq_error, sizeof(unsigned int));
    if (err != cudaSuccess || !clear) return err;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_seq_error, &zero, sizeof(unsigned int));
}

}  // namespace gq4

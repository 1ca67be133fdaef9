// gq4_stream.cu -- persistent, bulk-copy (TMA) fed CUDA-core kernels for the
// one-lane (M = 1) decode matvec family: plain, quad routing, RMSNorm
// prologue and SiLU-gated gate/up.
//
// Operation (gerbil moonshine-stt bundle, WGSL_QUAD_MATVEC_INT4 and
// WGSL_NORM_MATVEC_INT4; the DualMatVecInt4, GatedMatVecInt4 and
// SwiGLUGatedMatVecInt4 fusion docs): C[n] = sum_k a[k] * (q(n,k) - z) * s,
// a built by the call's prologue; two matrices for gate/up or dual.
//
// Decomposition.  At M = 1 the path is one streaming pass over the weights,
// so the kernel is organised around moving bytes:
//   * Persistent grid, one CTA per SM.  CTA b owns one contiguous range of
//     whole columns, balanced in units of 1, 2 or 4 columns so that every
//     copy of scale/zero rows starts 16-byte aligned.  Contiguous columns are
//     contiguous bytes in the [N][K/8] layout.
//   * One producer warp streams the range with cp.async.bulk (global ->
//     shared, completion on mbarriers): the CTA's scale and zero rows once,
//     at the start, then the packed codes through a ring of S stages.  A
//     stage holds the columns of WPS warp slots, one bulk copy per matrix:
//     few, large copies (the per-SM rate of bulk-copy requests, not bytes,
//     limits small copies).
//   * A warp slot is SPW whole columns (or SPW/2 gate and SPW/2 up columns).
//     Consumer warps take slots round-robin; a warp walks all of K for its
//     slot (lane l owns 32-code chunk groups l, l+32, ...) and reduces it
//     once with an xor reduce-scatter.  No cross-warp reduction, no group
//     barriers in the steady state.
//   * Activations are staged once per CTA in shared memory as 24-bit
//     fixed-point byte pieces with a power-of-two scale per chunk group,
//     arranged per packed word for dp4a and XOR-swizzled so that a warp's
//     128-bit loads are conflict-free (gq4_onelane.cuh); every activation
//     load serves all SPW streams.  The RMSNorm prologue stages x * W_norm
//     (x = A + A_b) and returns the inverse RMS, applied once to each
//     finished dot product.
//   * Per word, one logic operation and one add split the codes into even
//     and odd byte lanes and six dp4a accumulate them against the three
//     activation pieces, exactly in integers; per chunk group the integer
//     part of the zero point comes off through the piece sums and the
//     fractional part through the activation sum (see gq4_device.cuh).
//   * Every mbarrier wait is bounded in time; on expiry the kernel records
//     an error in a device word (gq4_device_error) and leaves.
#include <atomic>
#include <cstdint>

#include "gq4_device.cuh"
#include "gq4_host.h"
#include "gq4_internal.h"
#include "gq4_onelane.cuh"
#include "gq4_tma.cuh"

namespace gq4 {

// Sticky device-side error word (bit 0: a wait for a bulk copy timed out).
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kActBatch = 12;  // activation float4 per consumer thread per prologue batch
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 32;
constexpr uint32_t kSmemLimit = 220u * 1024u;

struct StreamParams {
    int K, N, gs;
    int KC, G;
    int KP;           // chunk groups per column (KC / R)
    int cps;          // columns per warp slot (per matrix)
    int wps;          // warp slots per stage
    int S;            // ring depth (stages)
    int unit;         // column granularity of the balanced split
    int n_units;
    int max_cols;     // most columns any CTA owns (sizes the scale/zero area)
    uint32_t stage_bytes;
    uint32_t off_w[2];              // within a stage
    uint32_t off_s[2], off_z[2];    // scale/zero rows of the CTA's range
    uint32_t off_act, off_norm, off_bar;
    unsigned long long group_magic;
    uint32_t magic_bits;  // 0x0F0F0F0F (even-code mask), read from the parameter bank
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

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Programmatic dependent launch (PTX griddepcontrol, sm_90 and later).
__device__ __forceinline__ void grid_dependents_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_arrive(int id, int threads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void record_error(unsigned int bits)
{
    atomicOr(&g_device_error, bits);
}

// R: consecutive 32-code chunks per chunk group (R = 2 only when a scale
// group holds at least 64 codes, so both chunks share one scale and zero).
// SPW: weight streams per warp per slot (columns, or gate and up columns).
template <int NMAT, int PRO, int EPI, int R, int SPW>
__global__ void __launch_bounds__(kThreads, 1)
stream_matvec_kernel(const __grid_constant__ StreamParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + kMaxStages;
    uint64_t *ready = empty + kMaxStages;  // consumers' prologue done
    uint64_t *srows = ready + 1;           // scale/zero rows landed
    // Sequence number of the stage a ring entry currently holds.  Entries are
    // shared by warps taking slots round-robin, so a warp first waits for its
    // stage's number (the previous occupant's barrier phase is then complete)
    // and only then for the barrier phase: a parity wait alone could match the
    // phase two steps back while the previous occupant is still landing.
    int *s_seq = reinterpret_cast<int *>(srows + 1);
    uint4 *s_act = reinterpret_cast<uint4 *>(smem + p.off_act);
    float *s_norm = reinterpret_cast<float *>(smem + p.off_norm);

    constexpr int CPS = NMAT == 2 ? SPW / 2 : SPW;  // columns per warp slot (per matrix)
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ctid = threadIdx.x;                   // consumer thread id (< kConsumerWarps*32)

    // ---- this CTA's column range (whole units) ----
    const int u0 = (int)((long long)p.n_units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)p.n_units * (blockIdx.x + 1) / gridDim.x);
    const int col_begin = u0 * p.unit;
    const int col_end = min(u1 * p.unit, p.N);
    if (col_begin >= col_end) return;  // uniform for the CTA, before any barrier
    const int ncols = col_end - col_begin;
    const int stage_cols = p.wps * CPS;
    const int n_stages = (ncols + stage_cols - 1) / stage_cols;
    const int n_slots = (ncols + CPS - 1) / CPS;

    // =====================================================================
    // Producer warp.  Its lane 0 initialises the mbarriers and starts
    // streaming at once; the consumers stage their activations meanwhile and
    // meet it at named barrier 2 only before their first mbarrier operation,
    // so neither waits for the other at the start.
    // =====================================================================
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            for (int s = 0; s < p.S; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], p.wps);
                s_seq[s] = -1;
            }
            mbar_init(ready, 1);
            mbar_init(srows, 1);
            mbar_fence_init();
        }
        __syncwarp();
        named_barrier_arrive(2, kThreads);
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            // scale and zero rows of the whole range: one copy per array (the
            // range starts 16-byte aligned; a ragged tail of the arrays, when
            // N*G is not a multiple of 4, is loaded plainly first)
            {
                const uint32_t s_all = (uint32_t)ncols * (uint32_t)p.G * 4u;
                const uint32_t s_bytes = s_all & ~15u;
                for (uint32_t b = s_bytes; b < s_all; b += 4) {
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        const size_t e = (size_t)col_begin * p.G + b / 4;
                        *reinterpret_cast<float *>(smem + p.off_s[m] + b) = p.scales[m][e];
                        *reinterpret_cast<float *>(smem + p.off_z[m] + b) = p.zeros[m][e];
                    }
                }
                mbar_arrive_expect_tx(srows, (uint32_t)NMAT * 2u * s_bytes);
                if (s_bytes) {
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        bulk_g2s(smem + p.off_s[m], p.scales[m] + (size_t)col_begin * p.G, s_bytes, srows);
                        bulk_g2s(smem + p.off_z[m], p.zeros[m] + (size_t)col_begin * p.G, s_bytes, srows);
                    }
                }
            }
            for (int i = 0; ok && i < n_stages; ++i) {
                const int slot = i % p.S;
                // Two stages go out at once; the rest wait for the consumers'
                // prologue, so its activation loads are not queued behind every
                // CTA's whole ring of weight copies.
                if (i == 2 && !mbar_wait(ready, 0)) {
                    record_error(1u);
                    ok = false;
                    break;
                }
                if (i >= p.S && !mbar_wait(&empty[slot], ((i / p.S) - 1) & 1)) {
                    record_error(1u);
                    ok = false;
                    break;
                }
                const int c0 = col_begin + i * stage_cols;
                const int nc = min(stage_cols, col_end - c0);
                const uint32_t w_bytes = (uint32_t)nc * (uint32_t)p.KC * 16u;
                unsigned char *dst = smem + (size_t)slot * p.stage_bytes;
                s_seq[slot] = i;  // published by the release of the arrive below
                mbar_arrive_expect_tx(&full[slot], (uint32_t)NMAT * w_bytes);
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
                    bulk_g2s(dst + p.off_w[m], p.Bq[m] + (size_t)c0 * p.KC, w_bytes, &full[slot]);
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
    // Consumer warps: prologue (activations into shared memory).
    // =====================================================================
    constexpr int kCT = kConsumerWarps * 32;
    // The activations may be the previous kernel's outputs: wait for that
    // grid to complete (its writes visible).  The producer does not wait: the
    // weights do not depend on it, so they stream in meanwhile.
    grid_dependency_wait();
    // inv: the norm prologue's inverse RMS, applied to each finished dot product
    const float inv = stage_activations_i8<R, PRO, kCT, kActBatch, LoadReadOnly>(
        p.K, p.A, p.A_b, p.W_norm, p.eps, p.residual_out, blockIdx.x == 0, s_act, s_norm, ctid, 1);
    named_barrier(2, kThreads);  // the producer has initialised the mbarriers
    if (ctid == 0) mbar_arrive(ready);

    // =====================================================================
    // Consumer warps: slots round-robin.
    // =====================================================================
    // A consumer whose bounded wait expires stops waiting and reading (its
    // outputs become NaN) but still releases its stages.
    bool failed = !mbar_wait(srows, 0);
    if (failed) record_error(1u);
    const uint32_t mask = p.magic_bits;
    const int swap = chunk_swap<R>(lane);
    const float *srow[NMAT];
    const float *zrow[NMAT];
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
        srow[m] = reinterpret_cast<const float *>(smem + p.off_s[m]);
        zrow[m] = reinterpret_cast<const float *>(smem + p.off_z[m]);
    }

    for (int i = warp; i < n_slots; i += kConsumerWarps) {
        // A warp starting its last slot lets the next kernel in the stream be
        // scheduled (once every CTA has done so or left): its CTAs then take
        // SMs as this grid's CTAs leave and start streaming their weights; it
        // reads this grid's outputs only after its own dependency wait.
        // Signalling at the start would let a third kernel queue for SMs
        // ahead of the second's.
        if (i + kConsumerWarps >= n_slots && lane == 0) grid_dependents_launch();
        const int stage = i / p.wps;
        const int sub = i - stage * p.wps;
        const int ring = stage % p.S;
        const int lc0 = i * CPS;  // first column of the slot, relative to col_begin
        const int nc = min(CPS, ncols - lc0);
        if (!failed &&
            !(wait_shared_eq(&s_seq[ring], stage) && mbar_wait(&full[ring], (stage / p.S) & 1))) {
            record_error(1u);
            failed = true;
        }
        const unsigned char *sl = smem + (size_t)ring * p.stage_bytes;

        float acc[SPW];
#pragma unroll
        for (int q = 0; q < SPW; ++q) acc[q] = 0.0f;

        // The slot's packed words of matrix `mat`, column `lc` (a short last
        // slot repeats its column 0, whose result is then discarded).
        auto slot_words = [&](int q) -> const uint4 * {
            const int mat = NMAT == 2 ? (q / CPS) : 0;
            int lc = NMAT == 2 ? (q % CPS) : q;
            lc = lc < nc ? lc : 0;
            return reinterpret_cast<const uint4 *>(sl + p.off_w[mat]) + (size_t)(sub * CPS + lc) * p.KC;
        };
        // One chunk group (R chunks) of all SPW streams.
        auto group_dot = [&](int jg, const uint4 (&wq)[SPW][R]) {
            const int grp = chunk_group(jg * R, p.group_magic);
            float sc[SPW], zz[SPW];
#pragma unroll
            for (int q = 0; q < SPW; ++q) {
                const int mat = NMAT == 2 ? (q / CPS) : 0;
                int lc = NMAT == 2 ? (q % CPS) : q;
                lc = lc < nc ? lc : 0;
                const int si = (lc0 + lc) * p.G + grp;
                sc[q] = srow[mat][si];
                zz[q] = zrow[mat][si];
            }
            chunk_group_dot_i8<SPW, R>(s_act, jg, swap, wq, sc, zz, mask, acc);
        };

        if (!failed) {
            for (int jg = lane; jg < p.KP; jg += 32) {
                uint4 wq[SPW][R];
#pragma unroll
                for (int q = 0; q < SPW; ++q) {
                    const uint4 *w = slot_words(q);
#pragma unroll
                    for (int r = 0; r < R; ++r) wq[q][r] = w[jg * R + (r ^ swap)];
                }
                group_dot(jg, wq);
            }
        }
        // this warp's part of the stage has been read: release it
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[ring]);

        // ---- reduce-scatter of the SPW streams across the warp ----
        float total;
        int q_of_lane;
        if constexpr (SPW == 4) {
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
            total = hi8 ? k1 : k0;
            total += __shfl_xor_sync(0xffffffffu, hi8 ? k0 : k1, 8);
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
            // lane 0 -> stream 0, lane 8 -> 1, lane 16 -> 2, lane 24 -> 3
            q_of_lane = ((lane >> 4) << 1) | ((lane >> 3) & 1);
        } else {
            // step 16: lanes < 16 keep stream 0, lanes >= 16 keep stream 1
            const bool hi16 = (lane & 16) != 0;
            total = hi16 ? acc[1] : acc[0];
            total += __shfl_xor_sync(0xffffffffu, hi16 ? acc[0] : acc[1], 16);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
            q_of_lane = lane >> 4;  // lane 0 -> stream 0, lane 16 -> stream 1
        }
        if constexpr (PRO == kProNorm) total *= inv;
        if (failed) total = __int_as_float(0x7fffffff);

        // ---- epilogue ----
        constexpr int kLaneStride = 32 / SPW;  // lanes holding one stream's total
        const int c0 = col_begin + lc0;
        if constexpr (EPI == kEpiGated) {
            // streams 0 .. CPS-1 are gate columns, CPS .. 2*CPS-1 the up columns
            const float u = __shfl_down_sync(0xffffffffu, total, 16);
            if ((lane % kLaneStride) == 0 && lane < 16) {
                const int lc = q_of_lane;
                if (lc < nc) {
                    const float gv = total;
                    p.out[0][c0 + lc] = gv / (1.0f + expf(-gv)) * u;
                }
            }
        } else if constexpr (EPI == kEpiDual) {
            // streams 0 .. CPS-1 are columns of matrix 0, CPS .. 2*CPS-1 of matrix 1
            if ((lane % kLaneStride) == 0) {
                const int mat = q_of_lane / CPS;
                const int lc = q_of_lane - mat * CPS;
                if (lc < nc) p.out[mat][c0 + lc] = total;
            }
        } else {
            if ((lane % kLaneStride) == 0) {
                const int lc = q_of_lane;
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
    if constexpr (PRO == kProNorm) {
        if (blockIdx.x == 0 && p.norm_out)
            write_norm_out<kCT, LoadReadOnly>(p.K, p.A, p.A_b, p.W_norm, inv, p.norm_out, ctid);
    }
}

template <int NMAT, int PRO, int EPI, int R, int SPW>
cudaError_t launch_stream_variant(const StreamParams &prm, size_t smem, cudaStream_t stream)
{
    auto kern = stream_matvec_kernel<NMAT, PRO, EPI, R, SPW>;
    int dev = 0, sms = 0;
    cudaError_t err;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    // Raise this kernel's dynamic shared-memory limit once per device (the
    // flags are per template instance: one kernel each).
    constexpr int kMaxDevices = 64;
    static std::atomic<unsigned char> smem_ready[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices || !smem_ready[dev].load(std::memory_order_acquire)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)(kSmemLimit + 4096u));
        if (err != cudaSuccess) return err;
        // every variant takes the same (largest) shared-memory carveout, so
        // an SM never has to drain to change it between consecutive calls
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   (int)cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < kMaxDevices) smem_ready[dev].store(1, std::memory_order_release);
    }
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    int grid = sms;
    if (grid > prm.n_units) grid = prm.n_units;
    // Launched with programmatic stream serialization: this kernel's CTAs may
    // start while the previous kernel in the stream finishes (its producer
    // then streams weights early); its consumers wait for that kernel's
    // completion before reading activations (griddepcontrol.wait).
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
cudaError_t launch_stream_rs(const StreamParams &prm, int R, int spw, size_t smem, cudaStream_t stream)
{
    if (R == 2)
        return spw == 4 ? launch_stream_variant<NMAT, PRO, EPI, 2, 4>(prm, smem, stream)
                        : launch_stream_variant<NMAT, PRO, EPI, 2, 2>(prm, smem, stream);
    return spw == 4 ? launch_stream_variant<NMAT, PRO, EPI, 1, 4>(prm, smem, stream)
                    : launch_stream_variant<NMAT, PRO, EPI, 1, 2>(prm, smem, stream);
}

// Ring geometry for a call; false when the call does not fit this path.
bool plan_stream(const Call &call, StreamParams &prm, int &R, int &spw, size_t &smem, int grid)
{
    prm.K = call.K;
    prm.N = call.N;
    prm.gs = call.gs;
    prm.KC = call.K / 32;
    prm.G = call.K / call.gs;
    // Long columns (K > 8192: few columns per CTA, 10+ chunk steps per
    // lane): single-chunk groups (the lanes' last step is nearly full), two
    // columns per slot (the CTA's slots fill the warps' rounds) and one slot
    // per stage (a warp's stage is released as soon as the warp is done).
    // Measured on the 11008-long down projection: 13.6 -> 10.2 us.
    const bool long_cols = call.K > 8192;
    // two consecutive chunks per chunk group when a scale group spans them
    // (the integer sums of a chunk group stay exact up to 64 codes)
    R = (call.gs >= 64 && prm.KC % 2 == 0) ? 2 : 1;
    prm.KP = prm.KC / R;
    prm.unit = 4 / gcd_int(prm.G, 4);
    prm.n_units = (call.N + prm.unit - 1) / prm.unit;
    if (grid > prm.n_units) grid = prm.n_units;
    prm.max_cols = ((prm.n_units + grid - 1) / grid) * prm.unit;
    const uint32_t act_bytes = round_up((uint32_t)prm.KC * 128u, 128u);
    const uint32_t rows_bytes = round_up((uint32_t)prm.max_cols * prm.G * 4u, 128u);
    const uint32_t fixed = act_bytes + 2u * call.nmat * rows_bytes + 128u +
                           (2 * kMaxStages + 2) * 8u + kMaxStages * 4u;
    const int spw_first = long_cols ? 2 : 4, spw_last = 2;
    // stage size cap (gate/up pairs: 24 KB, measured 16.1 -> 15.4 us on
    // 4096 -> 2 x 11008 against 48 KB; 12 KB is slower again)
    const uint32_t stage_cap = (long_cols ? 12u : call.nmat == 2 ? 24u : 48u) * 1024u;
    for (spw = spw_first; spw >= spw_last; spw /= 2) {
        const int cps = call.nmat == 2 ? spw / 2 : spw;
        // warp slots per stage: aim at ~32-48 KB per bulk copy round (long
        // columns: one slot)
        const uint32_t slot_bytes = (uint32_t)call.nmat * cps * prm.KC * 16u;
        for (int wps = kConsumerWarps; wps >= 1; wps /= 2) {
            const uint32_t stage = round_up(slot_bytes * wps, 128u);
            if (wps > 1 && stage > stage_cap) continue;
            // at least two stages (with fewer warp slots in the ring than
            // consumer warps, the extra warps simply wait their turn)
            if (fixed + stage * 2u > kSmemLimit) continue;
            int S = (int)((kSmemLimit - fixed) / stage);
            if (S > kMaxStages) S = kMaxStages;
            prm.S = S;
            prm.cps = cps;
            prm.wps = wps;
            prm.stage_bytes = stage;
            for (int m = 0; m < call.nmat; ++m) prm.off_w[m] = (uint32_t)m * cps * wps * prm.KC * 16u;
            uint32_t off = round_up((uint32_t)S * stage, 128u);
            for (int m = 0; m < call.nmat; ++m) {
                prm.off_s[m] = off;
                off += rows_bytes;
                prm.off_z[m] = off;
                off += rows_bytes;
            }
            prm.off_act = off;
            prm.off_norm = prm.off_act + act_bytes;
            prm.off_bar = prm.off_norm + 128u;
            smem = prm.off_bar + (2 * kMaxStages + 2) * sizeof(uint64_t) + kMaxStages * sizeof(int);
            return smem <= kSmemLimit + 4096u;
        }
    }
    return false;
}

int sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace

bool stream_path_supported(const Call &call)
{
    if (call.M != 1) return false;
    for (int m = 0; m < call.nmat; ++m) {
        if ((reinterpret_cast<uintptr_t>(call.scales[m]) & 15u) != 0) return false;
        if ((reinterpret_cast<uintptr_t>(call.zeros[m]) & 15u) != 0) return false;
    }
    StreamParams prm{};
    int R, spw;
    size_t smem;
    const int sms = sm_count();
    return sms > 0 && plan_stream(call, prm, R, spw, smem, sms);
}

cudaError_t launch_stream(const Call &call, cudaStream_t stream)
{
    StreamParams prm{};
    int R = 1, spw = 4;
    size_t smem = 0;
    const int sms = sm_count();
    if (sms <= 0 || !plan_stream(call, prm, R, spw, smem, sms)) return cudaErrorInvalidValue;
    const unsigned long long cpgrp = (unsigned long long)(call.gs / 32);
    prm.group_magic = ((1ull << 40) + cpgrp - 1) / cpgrp;
    prm.magic_bits = 0x0F0F0F0Fu;
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
        case kProNorm: return launch_stream_rs<1, kProNorm, kEpiStore>(prm, R, spw, smem, stream);
        case kProSigmoid: return launch_stream_rs<1, kProSigmoid, kEpiStore>(prm, R, spw, smem, stream);
        case kProSwiglu: return launch_stream_rs<1, kProSwiglu, kEpiStore>(prm, R, spw, smem, stream);
        default: return launch_stream_rs<1, kProNone, kEpiStore>(prm, R, spw, smem, stream);
        }
    case kEpiQuad:
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_stream_rs<1, kProNone, kEpiQuad>(prm, R, spw, smem, stream);
    case kEpiGated:
        if (pro == kProNorm) return launch_stream_rs<2, kProNorm, kEpiGated>(prm, R, spw, smem, stream);
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_stream_rs<2, kProNone, kEpiGated>(prm, R, spw, smem, stream);
    case kEpiDual:
        if (pro != kProNone) return cudaErrorInvalidValue;
        return launch_stream_rs<2, kProNone, kEpiDual>(prm, R, spw, smem, stream);
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

// gq4_api.cu -- the extern "C" entry points of libgq4 (declared in gq4.h).
//
// Every entry point validates its arguments on the host, synchronously,
// before anything is enqueued; a non-OK status means the stream is untouched.
// The checks mirror the pages' preconditions: the quad and norm fusion passes
// of the gerbil executor refuse to fuse when an output buffer aliases an
// input or another output (fuseMambaFrontDecodeEntries,
// fuseNormMatVecDecodeEntries), and the WGSL kernels assume K and the group
// size are whole multiples of the 32-code vec4u load.
#include <cstdint>
#include <cstring>
#include <vector>

#include "gq4.h"
#include "gq4_internal.h"

namespace {

constexpr int kMaxK = 1 << 24;  // keeps 32-code chunk indices below 2^20

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void *p, size_t bytes)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + bytes};
}

bool overlap(Range a, Range b)
{
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Collects the byte ranges of a call and checks them.
struct RangeSet {
    Range in[16];
    int n_in = 0;
    Range out[8];
    int n_out = 0;
    void input(const void *p, size_t bytes)
    {
        if (p && bytes) in[n_in++] = range_of(p, bytes);
    }
    void output(const void *p, size_t bytes)
    {
        if (p && bytes) out[n_out++] = range_of(p, bytes);
    }
    bool disjoint() const
    {
        for (int i = 0; i < n_out; ++i) {
            for (int j = 0; j < n_in; ++j)
                if (overlap(out[i], in[j])) return false;
            for (int j = i + 1; j < n_out; ++j)
                if (overlap(out[i], out[j])) return false;
        }
        return true;
    }
};

gq4_status check_shape(int M, int K, int N, int gs)
{
    if (M < 1 || M > GQ4_MAX_LANES) return GQ4_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || gs <= 0) return GQ4_ERR_INVALID_ARG;
    if (K > kMaxK) return GQ4_ERR_INVALID_ARG;
    if (gs % 32 != 0 || K % gs != 0) return GQ4_ERR_INVALID_ARG;
    return GQ4_OK;
}

// One int4 matrix: pointers present, Bq 16-byte aligned, scales/zeros 4-byte.
gq4_status check_weights(const uint32_t *Bq, const float *s, const float *z, int K, int N, int gs,
                         RangeSet &rs)
{
    if (!Bq || !s || !z) return GQ4_ERR_INVALID_ARG;
    if (!aligned(Bq, 16) || !aligned(s, 4) || !aligned(z, 4)) return GQ4_ERR_MISALIGNED;
    const size_t n = (size_t)N;
    rs.input(Bq, n * (size_t)K / 2);
    rs.input(s, n * (size_t)(K / gs) * sizeof(float));
    rs.input(z, n * (size_t)(K / gs) * sizeof(float));
    return GQ4_OK;
}

gq4_status check_norm(const gq4_norm *norm, int M, int K, RangeSet &rs)
{
    if (!norm->W_norm) return GQ4_ERR_INVALID_ARG;
    if (!(norm->eps >= 0.0f)) return GQ4_ERR_INVALID_ARG;  // also rejects NaN
    const size_t mk = (size_t)M * (size_t)K * sizeof(float);
    if (!aligned(norm->W_norm, 16) || (norm->A_b && !aligned(norm->A_b, 16)) ||
        (norm->residual_out && !aligned(norm->residual_out, 16)) ||
        (norm->norm_out && !aligned(norm->norm_out, 16)))
        return GQ4_ERR_MISALIGNED;
    rs.input(norm->A_b, mk);
    rs.input(norm->W_norm, (size_t)K * sizeof(float));
    rs.output(norm->residual_out, mk);
    rs.output(norm->norm_out, mk);
    return GQ4_OK;
}

gq4_status check_activation(const float *A, int M, int K, RangeSet &rs)
{
    if (!A) return GQ4_ERR_INVALID_ARG;
    if (!aligned(A, 16)) return GQ4_ERR_MISALIGNED;
    rs.input(A, (size_t)M * (size_t)K * sizeof(float));
    return GQ4_OK;
}

gq4_status check_output(const float *out, size_t elems, RangeSet &rs)
{
    if (elems == 0) return GQ4_OK;
    if (!out) return GQ4_ERR_INVALID_ARG;
    if (!aligned(out, 4)) return GQ4_ERR_MISALIGNED;
    rs.output(out, elems * sizeof(float));
    return GQ4_OK;
}

#define GQ4_TRY(expr)                       \
    do {                                    \
        const gq4_status st_ = (expr);      \
        if (st_ != GQ4_OK) return st_;      \
    } while (0)

gq4_status run(const gq4::Call &call, cudaStream_t stream)
{
    // one lane: the persistent streaming kernel; 2..4 lanes: the persistent
    // warp-MMA kernel; 16..32 lanes: the bf16 tensor-core kernel; otherwise
    // (and for shapes those do not take) the fp32 CUDA-core kernel
    cudaError_t err;
    if (gq4::stream_path_supported(call))
        err = gq4::launch_stream(call, stream);
    else if (gq4::lanes_path_supported(call))
        err = gq4::launch_lanes(call, stream);
    else if (gq4::tc_path_supported(call))
        err = gq4::launch_tc(call, stream);
    else
        err = gq4::launch_fp32(call, stream);
    return err == cudaSuccess ? GQ4_OK : GQ4_ERR_CUDA;
}

gq4::Call base_call(int M, int K, int N, int gs, const float *A)
{
    gq4::Call c;
    std::memset(&c, 0, sizeof(c));
    c.M = M;
    c.K = K;
    c.N = N;
    c.gs = gs;
    c.A = A;
    c.nmat = 1;
    c.seg_start[0] = 0;
    c.seg_start[1] = c.seg_start[2] = c.seg_start[3] = N;
    c.seg_len[0] = N;
    return c;
}

// Validation and the internal call of each entry point (shared with the
// call sequences).

gq4_status build_matvec(int M, int K, int N, int group_size, const float *A, const uint32_t *Bq,
                        const float *scales, const float *zeros, float *C, gq4::Call &call)
{
    GQ4_TRY(check_shape(M, K, N, group_size));
    RangeSet rs;
    GQ4_TRY(check_activation(A, M, K, rs));
    GQ4_TRY(check_weights(Bq, scales, zeros, K, N, group_size, rs));
    if (!C) return GQ4_ERR_INVALID_ARG;
    GQ4_TRY(check_output(C, (size_t)M * (size_t)N, rs));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;

    call = base_call(M, K, N, group_size, A);
    call.Bq[0] = Bq;
    call.scales[0] = scales;
    call.zeros[0] = zeros;
    call.epi = gq4::kEpiStore;
    call.out[0] = C;
    return GQ4_OK;
}

gq4_status build_quad(int M, int K, int N, int group_size, int n0, int n1, int n2, const float *A,
                      const uint32_t *Bq, const float *scales, const float *zeros, float *const outs[4],
                      gq4::Call &call)
{
    GQ4_TRY(check_shape(M, K, N, group_size));
    if (!(0 <= n0 && n0 <= n1 && n1 <= n2 && n2 <= N)) return GQ4_ERR_INVALID_ARG;
    RangeSet rs;
    GQ4_TRY(check_activation(A, M, K, rs));
    GQ4_TRY(check_weights(Bq, scales, zeros, K, N, group_size, rs));
    const int start[4] = {0, n0, n1, n2};
    const int len[4] = {n0, n1 - n0, n2 - n1, N - n2};
    for (int i = 0; i < 4; ++i) GQ4_TRY(check_output(outs[i], (size_t)M * (size_t)len[i], rs));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;

    call = base_call(M, K, N, group_size, A);
    call.Bq[0] = Bq;
    call.scales[0] = scales;
    call.zeros[0] = zeros;
    call.epi = gq4::kEpiQuad;
    for (int i = 0; i < 4; ++i) {
        call.out[i] = outs[i];
        call.seg_start[i] = start[i];
        call.seg_len[i] = len[i];
    }
    return GQ4_OK;
}

gq4_status build_norm(int M, int K, int N, int group_size, const gq4_norm *norm, const float *A,
                      const uint32_t *Bq, const float *scales, const float *zeros, float *C,
                      gq4::Call &call)
{
    GQ4_TRY(check_shape(M, K, N, group_size));
    if (!norm) return GQ4_ERR_INVALID_ARG;
    RangeSet rs;
    GQ4_TRY(check_activation(A, M, K, rs));
    GQ4_TRY(check_norm(norm, M, K, rs));
    GQ4_TRY(check_weights(Bq, scales, zeros, K, N, group_size, rs));
    if (!C) return GQ4_ERR_INVALID_ARG;
    GQ4_TRY(check_output(C, (size_t)M * (size_t)N, rs));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;

    call = base_call(M, K, N, group_size, A);
    call.norm = norm;
    call.Bq[0] = Bq;
    call.scales[0] = scales;
    call.zeros[0] = zeros;
    call.epi = gq4::kEpiStore;
    call.out[0] = C;
    return GQ4_OK;
}

gq4_status build_gated(int M, int K, int N, int group_size, const gq4_norm *norm, const float *A,
                       const uint32_t *Bq_gate, const float *scales_gate, const float *zeros_gate,
                       const uint32_t *Bq_up, const float *scales_up, const float *zeros_up,
                       float *out, gq4::Call &call)
{
    GQ4_TRY(check_shape(M, K, N, group_size));
    RangeSet rs;
    GQ4_TRY(check_activation(A, M, K, rs));
    if (norm) GQ4_TRY(check_norm(norm, M, K, rs));
    GQ4_TRY(check_weights(Bq_gate, scales_gate, zeros_gate, K, N, group_size, rs));
    GQ4_TRY(check_weights(Bq_up, scales_up, zeros_up, K, N, group_size, rs));
    if (!out) return GQ4_ERR_INVALID_ARG;
    GQ4_TRY(check_output(out, (size_t)M * (size_t)N, rs));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;

    call = base_call(M, K, N, group_size, A);
    call.norm = norm;
    call.nmat = 2;
    call.Bq[0] = Bq_gate;
    call.scales[0] = scales_gate;
    call.zeros[0] = zeros_gate;
    call.Bq[1] = Bq_up;
    call.scales[1] = scales_up;
    call.zeros[1] = zeros_up;
    call.epi = gq4::kEpiGated;
    call.out[0] = out;
    return GQ4_OK;
}

// One call of a sequence (M = 1).
gq4_status build_seq_call(const gq4_call &c, gq4::Call &call)
{
    switch (c.op) {
    case GQ4_OP_MATVEC:
        return build_matvec(1, c.K, c.N, c.group_size, c.A, c.Bq[0], c.scales[0], c.zeros[0], c.out[0],
                            call);
    case GQ4_OP_QUAD:
        return build_quad(1, c.K, c.N, c.group_size, c.n0, c.n1, c.n2, c.A, c.Bq[0], c.scales[0],
                          c.zeros[0], c.out, call);
    case GQ4_OP_NORM:
        if (!c.has_norm) return GQ4_ERR_INVALID_ARG;
        return build_norm(1, c.K, c.N, c.group_size, &c.norm, c.A, c.Bq[0], c.scales[0], c.zeros[0],
                          c.out[0], call);
    case GQ4_OP_GATED:
        return build_gated(1, c.K, c.N, c.group_size, c.has_norm ? &c.norm : nullptr, c.A, c.Bq[0],
                           c.scales[0], c.zeros[0], c.Bq[1], c.scales[1], c.zeros[1], c.out[0], call);
    default:
        return GQ4_ERR_INVALID_ARG;
    }
}

gq4_status build_dual(int M, int K, int N, int group_size, const float *A, const uint32_t *Bq0,
                      const float *scales0, const float *zeros0, const uint32_t *Bq1,
                      const float *scales1, const float *zeros1, float *C0, float *C1,
                      gq4::Call &call)
{
    GQ4_TRY(check_shape(M, K, N, group_size));
    RangeSet rs;
    GQ4_TRY(check_activation(A, M, K, rs));
    GQ4_TRY(check_weights(Bq0, scales0, zeros0, K, N, group_size, rs));
    GQ4_TRY(check_weights(Bq1, scales1, zeros1, K, N, group_size, rs));
    if (!C0 || !C1) return GQ4_ERR_INVALID_ARG;
    GQ4_TRY(check_output(C0, (size_t)M * (size_t)N, rs));
    GQ4_TRY(check_output(C1, (size_t)M * (size_t)N, rs));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;

    call = base_call(M, K, N, group_size, A);
    call.nmat = 2;
    call.Bq[0] = Bq0;
    call.scales[0] = scales0;
    call.zeros[0] = zeros0;
    call.Bq[1] = Bq1;
    call.scales[1] = scales1;
    call.zeros[1] = zeros1;
    call.epi = gq4::kEpiDual;
    call.out[0] = C0;
    call.out[1] = C1;
    return GQ4_OK;
}

gq4_status build_gated_input(int M, int K, int N, int group_size, int kind, const float *X,
                             const float *G, const uint32_t *Bq, const float *scales,
                             const float *zeros, float *C, gq4::Call &call)
{
    GQ4_TRY(check_shape(M, K, N, group_size));
    RangeSet rs;
    GQ4_TRY(check_activation(X, M, K, rs));
    GQ4_TRY(check_activation(G, M, K, rs));
    GQ4_TRY(check_weights(Bq, scales, zeros, K, N, group_size, rs));
    if (!C) return GQ4_ERR_INVALID_ARG;
    GQ4_TRY(check_output(C, (size_t)M * (size_t)N, rs));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;

    call = base_call(M, K, N, group_size, X);
    call.gate_kind = kind;
    call.G = G;
    call.Bq[0] = Bq;
    call.scales[0] = scales;
    call.zeros[0] = zeros;
    call.epi = gq4::kEpiStore;
    call.out[0] = C;
    return GQ4_OK;
}

}  // namespace

extern "C" {

gq4_status gq4_matvec(int M, int K, int N, int group_size, const float *A, const uint32_t *Bq,
                      const float *scales, const float *zeros, float *C, cudaStream_t stream)
{
    gq4::Call call;
    GQ4_TRY(build_matvec(M, K, N, group_size, A, Bq, scales, zeros, C, call));
    return run(call, stream);
}

gq4_status gq4_quad_matvec(int M, int K, int N, int group_size, int n0, int n1, int n2,
                           const float *A, const uint32_t *Bq, const float *scales,
                           const float *zeros, float *out0, float *out1, float *out2,
                           float *out3, cudaStream_t stream)
{
    float *const outs[4] = {out0, out1, out2, out3};
    gq4::Call call;
    GQ4_TRY(build_quad(M, K, N, group_size, n0, n1, n2, A, Bq, scales, zeros, outs, call));
    return run(call, stream);
}

gq4_status gq4_norm_matvec(int M, int K, int N, int group_size, const gq4_norm *norm,
                           const float *A, const uint32_t *Bq, const float *scales,
                           const float *zeros, float *C, cudaStream_t stream)
{
    gq4::Call call;
    GQ4_TRY(build_norm(M, K, N, group_size, norm, A, Bq, scales, zeros, C, call));
    return run(call, stream);
}

gq4_status gq4_dual_matvec(int M, int K, int N, int group_size, const float *A,
                           const uint32_t *Bq0, const float *scales0, const float *zeros0,
                           const uint32_t *Bq1, const float *scales1, const float *zeros1,
                           float *C0, float *C1, cudaStream_t stream)
{
    gq4::Call call;
    GQ4_TRY(build_dual(M, K, N, group_size, A, Bq0, scales0, zeros0, Bq1, scales1, zeros1, C0, C1,
                       call));
    return run(call, stream);
}

gq4_status gq4_sigmoid_gated_matvec(int M, int K, int N, int group_size, const float *X,
                                    const float *G, const uint32_t *Bq, const float *scales,
                                    const float *zeros, float *C, cudaStream_t stream)
{
    gq4::Call call;
    GQ4_TRY(build_gated_input(M, K, N, group_size, gq4::kGateSigmoid, X, G, Bq, scales, zeros, C, call));
    return run(call, stream);
}

gq4_status gq4_swiglu_gated_matvec(int M, int K, int N, int group_size, const float *X,
                                   const float *G, const uint32_t *Bq, const float *scales,
                                   const float *zeros, float *C, cudaStream_t stream)
{
    gq4::Call call;
    GQ4_TRY(build_gated_input(M, K, N, group_size, gq4::kGateSwiglu, X, G, Bq, scales, zeros, C, call));
    return run(call, stream);
}

gq4_status gq4_gated_matvec(int M, int K, int N, int group_size, const gq4_norm *norm,
                            const float *A, const uint32_t *Bq_gate, const float *scales_gate,
                            const float *zeros_gate, const uint32_t *Bq_up,
                            const float *scales_up, const float *zeros_up, float *out,
                            cudaStream_t stream)
{
    gq4::Call call;
    GQ4_TRY(build_gated(M, K, N, group_size, norm, A, Bq_gate, scales_gate, zeros_gate, Bq_up,
                        scales_up, zeros_up, out, call));
    return run(call, stream);
}

size_t gq4_sequence_workspace_bytes(void)
{
    return gq4::kSeqWorkspaceBytes;
}

}  // extern "C"

namespace {

// Validates a call list against the launch scratch `scratch` (bytes
// [scratch, scratch + kSeqWorkspaceBytes) must not overlap any call's
// buffers) and builds the calls.  `persistent` tells whether the list runs
// as one persistent launch (every call plannable, scale/zero rows 16-byte
// aligned) or call by call.  Nothing is enqueued.
gq4_status prepare_sequence(const gq4_call *calls, int n_calls, const void *scratch,
                            std::vector<gq4::Call> &built, bool &persistent)
{
    built.assign((size_t)n_calls, gq4::Call{});
    persistent = true;
    for (int i = 0; i < n_calls; ++i) {
        GQ4_TRY(build_seq_call(calls[i], built[(size_t)i]));
        const gq4::Call &c = built[(size_t)i];
        const size_t mk = (size_t)c.M * (size_t)c.K * sizeof(float);
        // the scratch is the launch's own: no call may touch it
        RangeSet rs;
        rs.input(c.A, mk);
        for (int m = 0; m < c.nmat; ++m) {
            rs.input(c.Bq[m], (size_t)c.N * (size_t)c.K / 2);
            rs.input(c.scales[m], (size_t)c.N * (size_t)(c.K / c.gs) * sizeof(float));
            rs.input(c.zeros[m], (size_t)c.N * (size_t)(c.K / c.gs) * sizeof(float));
        }
        for (int j = 0; j < 4; ++j) rs.input(c.out[j], (size_t)c.M * (size_t)c.seg_len[j] * sizeof(float));
        if (c.norm) {
            rs.input(c.norm->A_b, mk);
            rs.input(c.norm->W_norm, (size_t)c.K * sizeof(float));
            rs.input(c.norm->residual_out, mk);
            rs.input(c.norm->norm_out, mk);
        }
        rs.output(scratch, gq4::kSeqWorkspaceBytes);
        if (!rs.disjoint()) return GQ4_ERR_ALIAS;
        // the persistent kernel copies scale/zero rows in bulk (16-byte bases)
        for (int m = 0; m < c.nmat; ++m)
            if (!aligned(c.scales[m], 16) || !aligned(c.zeros[m], 16)) persistent = false;
    }
    if (persistent) persistent = gq4::sequence_plannable(built.data(), n_calls);
    return GQ4_OK;
}

gq4_status run_prepared(const std::vector<gq4::Call> &built, bool persistent, void *scratch,
                        cudaStream_t stream)
{
    if (persistent)
        return gq4::launch_sequence(built.data(), (int)built.size(), scratch, stream) == cudaSuccess
                   ? GQ4_OK
                   : GQ4_ERR_CUDA;
    // otherwise the calls run one by one (same semantics, stream order)
    for (const gq4::Call &c : built) GQ4_TRY(run(c, stream));
    return GQ4_OK;
}

}  // namespace

extern "C" {

gq4_status gq4_run_sequence(const gq4_call *calls, int n_calls, void *workspace, cudaStream_t stream)
{
    if (n_calls < 0 || (n_calls > 0 && !calls)) return GQ4_ERR_INVALID_ARG;
    if (n_calls == 0) return GQ4_OK;
    if (!workspace) return GQ4_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return GQ4_ERR_MISALIGNED;
    std::vector<gq4::Call> built;
    bool persistent = false;
    GQ4_TRY(prepare_sequence(calls, n_calls, workspace, built, persistent));
    return run_prepared(built, persistent, workspace, stream);
}

gq4_status gq4_sequence_launches(const gq4_call *calls, int n_calls, int *launches)
{
    if (!launches || n_calls < 0 || (n_calls > 0 && !calls)) return GQ4_ERR_INVALID_ARG;
    *launches = 0;
    if (n_calls == 0) return GQ4_OK;
    std::vector<gq4::Call> built;
    bool persistent = false;
    GQ4_TRY(prepare_sequence(calls, n_calls, nullptr, built, persistent));
    if (persistent) *launches = (n_calls + gq4::kSeqMaxCalls - 1) / gq4::kSeqMaxCalls;
    return GQ4_OK;
}

gq4_status gq4_run_sequence_static(const gq4_call *calls, int n_calls, cudaStream_t stream)
{
    if (n_calls < 0 || (n_calls > 0 && !calls)) return GQ4_ERR_INVALID_ARG;
    if (n_calls == 0) return GQ4_OK;
    // the launch's scratch must fit the static array
    const size_t need = gq4::kSeqWorkspaceBytes;
    if (need > gq4::seq_static_scratch_bytes()) return GQ4_ERR_INVALID_ARG;
    void *scratch = nullptr;
    if (gq4::seq_static_scratch(&scratch) != cudaSuccess) return GQ4_ERR_CUDA;
    // every check runs before anything is enqueued
    std::vector<gq4::Call> built;
    bool persistent = false;
    GQ4_TRY(prepare_sequence(calls, n_calls, scratch, built, persistent));
    // what must start at zero (the barrier counters), only for the
    // persistent launch that uses them
    if (persistent && cudaMemsetAsync(scratch, 0, need, stream) != cudaSuccess) return GQ4_ERR_CUDA;
    return run_prepared(built, persistent, scratch, stream);
}

gq4_status gq4_unpack(int K, int N, const uint32_t *Bq, uint8_t *q, cudaStream_t stream)
{
    if (K <= 0 || N <= 0 || K % 32 != 0 || K > kMaxK) return GQ4_ERR_INVALID_ARG;
    if (!Bq || !q) return GQ4_ERR_INVALID_ARG;
    if (!aligned(Bq, 16) || !aligned(q, 4)) return GQ4_ERR_MISALIGNED;
    const size_t nk = (size_t)N * (size_t)K;
    if (overlap(range_of(Bq, nk / 2), range_of(q, nk))) return GQ4_ERR_ALIAS;
    return gq4::launch_unpack(K, N, Bq, q, stream) == cudaSuccess ? GQ4_OK : GQ4_ERR_CUDA;
}

gq4_status gq4_dequant(int K, int N, int group_size, const uint32_t *Bq, const float *scales,
                       const float *zeros, float *W, cudaStream_t stream)
{
    GQ4_TRY(check_shape(1, K, N, group_size));
    RangeSet rs;
    GQ4_TRY(check_weights(Bq, scales, zeros, K, N, group_size, rs));
    if (!W) return GQ4_ERR_INVALID_ARG;
    if (!aligned(W, 4)) return GQ4_ERR_MISALIGNED;
    rs.output(W, (size_t)N * (size_t)K * sizeof(float));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;
    return gq4::launch_dequant(K, N, group_size, Bq, scales, zeros, W, stream) == cudaSuccess
               ? GQ4_OK
               : GQ4_ERR_CUDA;
}

size_t gq4_gemm_workspace_bytes(int M, int K)
{
    if (M < 1 || K < 1) return 0;
    return gq4::gemm_workspace_bytes(M, K);
}

gq4_status gq4_gemm(int M, int K, int N, int group_size, const float *A, const uint32_t *Bq,
                    const float *scales, const float *zeros, float *C, void *workspace,
                    size_t workspace_bytes, cudaStream_t stream)
{
    if (M < 1 || M > GQ4_MAX_GEMM_ROWS) return GQ4_ERR_INVALID_ARG;
    GQ4_TRY(check_shape(1, K, N, group_size));
    RangeSet rs;
    GQ4_TRY(check_activation(A, M, K, rs));
    GQ4_TRY(check_weights(Bq, scales, zeros, K, N, group_size, rs));
    if (!C) return GQ4_ERR_INVALID_ARG;
    GQ4_TRY(check_output(C, (size_t)M * (size_t)N, rs));
    const size_t need = gq4::gemm_workspace_bytes(M, K);
    const bool use_ws = workspace && workspace_bytes >= need;
    if (use_ws) {
        if (!aligned(workspace, 256)) return GQ4_ERR_MISALIGNED;
        rs.output(workspace, need);
    }
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;
    if (M > 32 && use_ws && gq4::gemm_path_supported(K, N, group_size, scales, zeros))
        return gq4::launch_gemm(M, K, N, group_size, A, Bq, scales, zeros, C, workspace, stream) ==
                       cudaSuccess
                   ? GQ4_OK
                   : GQ4_ERR_CUDA;
    // chunks of up to 32 rows on the tensor-core kernel, in order on the
    // stream (the chunks only read the weights, so the programmatic launch of
    // one chunk while the previous finishes is safe)
    for (int m0 = 0; m0 < M; m0 += 32) {
        const int rows = M - m0 < 32 ? M - m0 : 32;
        gq4::Call call = base_call(rows, K, N, group_size, A + (size_t)m0 * K);
        call.Bq[0] = Bq;
        call.scales[0] = scales;
        call.zeros[0] = zeros;
        call.epi = gq4::kEpiStore;
        call.out[0] = C + (size_t)m0 * N;
        cudaError_t err;
        if (gq4::tc_rows_supported(call))
            err = gq4::launch_tc(call, stream);
        else if (rows == 1 && gq4::stream_path_supported(call))
            err = gq4::launch_stream(call, stream);
        else if (gq4::lanes_path_supported(call))
            err = gq4::launch_lanes(call, stream);
        else
            err = gq4::launch_fp32(call, stream);
        if (err != cudaSuccess) return GQ4_ERR_CUDA;
    }
    return GQ4_OK;
}

gq4_status gq4_quantize(int K, int N, int group_size, const float *W, uint32_t *Bq,
                        float *scales, float *zeros, cudaStream_t stream)
{
    GQ4_TRY(check_shape(1, K, N, group_size));
    if (!W || !Bq || !scales || !zeros) return GQ4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(Bq, 16) || !aligned(scales, 4) || !aligned(zeros, 4))
        return GQ4_ERR_MISALIGNED;
    const size_t n = (size_t)N, groups = n * (size_t)(K / group_size);
    RangeSet rs;
    rs.input(W, n * (size_t)K * sizeof(float));
    rs.output(Bq, n * (size_t)K / 2);
    rs.output(scales, groups * sizeof(float));
    rs.output(zeros, groups * sizeof(float));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;
    return gq4::launch_quantize(K, N, group_size, W, Bq, scales, zeros, stream) == cudaSuccess
               ? GQ4_OK
               : GQ4_ERR_CUDA;
}

gq4_status gq4_from_mlx(int K, int N, int group_size, const uint32_t *packed,
                        const float *mlx_scales, const float *mlx_biases, uint32_t *Bq,
                        float *scales, float *zeros, cudaStream_t stream)
{
    GQ4_TRY(check_shape(1, K, N, group_size));
    if (!packed || !mlx_scales || !mlx_biases || !Bq || !scales || !zeros)
        return GQ4_ERR_INVALID_ARG;
    if (!aligned(packed, 16) || !aligned(Bq, 16) || !aligned(mlx_scales, 4) ||
        !aligned(mlx_biases, 4) || !aligned(scales, 4) || !aligned(zeros, 4))
        return GQ4_ERR_MISALIGNED;
    const size_t n = (size_t)N, groups = n * (size_t)(K / group_size);
    RangeSet rs;
    // in place: Bq is packed itself (each word is read and written by one thread)
    if (packed != Bq) rs.input(packed, n * (size_t)K / 2);
    rs.input(mlx_scales, groups * sizeof(float));
    rs.input(mlx_biases, groups * sizeof(float));
    rs.output(Bq, n * (size_t)K / 2);
    rs.output(scales, groups * sizeof(float));
    rs.output(zeros, groups * sizeof(float));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;
    return gq4::launch_from_mlx(K, N, group_size, packed, mlx_scales, mlx_biases, Bq, scales,
                                zeros, stream) == cudaSuccess
               ? GQ4_OK
               : GQ4_ERR_CUDA;
}

gq4_status gq4_embedding(int T, int K, int V, int group_size, const int32_t *ids,
                         const uint32_t *Bq, const float *scales, const float *zeros, float *out,
                         cudaStream_t stream)
{
    if (T < 0) return GQ4_ERR_INVALID_ARG;
    GQ4_TRY(check_shape(1, K, V, group_size));
    RangeSet rs;
    GQ4_TRY(check_weights(Bq, scales, zeros, K, V, group_size, rs));
    if (T == 0) return GQ4_OK;
    if (!ids || !out) return GQ4_ERR_INVALID_ARG;
    if (!aligned(ids, 4) || !aligned(out, 16)) return GQ4_ERR_MISALIGNED;
    rs.input(ids, (size_t)T * sizeof(int32_t));
    rs.output(out, (size_t)T * (size_t)K * sizeof(float));
    if (!rs.disjoint()) return GQ4_ERR_ALIAS;
    return gq4::launch_embedding(T, K, V, group_size, ids, Bq, scales, zeros, out, stream) ==
                   cudaSuccess
               ? GQ4_OK
               : GQ4_ERR_CUDA;
}

gq4_status gq4_device_error(unsigned int *bits, int clear)
{
    if (!bits) return GQ4_ERR_INVALID_ARG;
    unsigned int a = 0, b = 0, c = 0, d = 0, e = 0;
    if (gq4::read_device_error(&a, clear != 0) != cudaSuccess) return GQ4_ERR_CUDA;
    if (gq4::read_tc_device_error(&b, clear != 0) != cudaSuccess) return GQ4_ERR_CUDA;
    if (gq4::read_seq_device_error(&c, clear != 0) != cudaSuccess) return GQ4_ERR_CUDA;
    if (gq4::read_quant_device_error(&d, clear != 0) != cudaSuccess) return GQ4_ERR_CUDA;
    if (gq4::read_embed_device_error(&e, clear != 0) != cudaSuccess) return GQ4_ERR_CUDA;
    unsigned int f = 0, l = 0;
    if (gq4::read_gemm_device_error(&f, clear != 0) != cudaSuccess) return GQ4_ERR_CUDA;
    if (gq4::read_lanes_device_error(&l, clear != 0) != cudaSuccess) return GQ4_ERR_CUDA;
    *bits = a | b | c | d | e | f | l;
    return GQ4_OK;
}

const char *gq4_status_string(gq4_status status)
{
    switch (status) {
    case GQ4_OK: return "ok";
    case GQ4_ERR_INVALID_ARG: return "invalid argument";
    case GQ4_ERR_UNSUPPORTED: return "unsupported";
    case GQ4_ERR_ALIAS: return "output overlaps an input or another output";
    case GQ4_ERR_CUDA: return "CUDA launch error";
    case GQ4_ERR_MISALIGNED: return "misaligned pointer";
    }
    return "unknown status";
}

int gq4_version(void)
{
    return 100;  // 0.1.0
}

}  // extern "C"

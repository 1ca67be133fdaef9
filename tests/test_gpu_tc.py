"""GPU parity of the batched-lane (16..32 lanes) bf16 tensor-core path.

Weights and activations are rounded to bf16 and multiplied on the tensor core
with f32 accumulation, so outputs are compared against the oracle under
|gpu - ref| <= 2e-2 * sum_k |a_k w_k| + 1e-6 (the RMSNorm side outputs stay
f32 and keep their f32 bounds).  Cases cover the 7B-shaped stack's four calls
at 16 and 32 lanes, ragged K (a final partial 256-code stage), ragged N
(partial tiles), group sizes 32..1024 including one that does not divide the
stage, scale rows that are not 16-byte multiples (read as super-rows of 2 or 4
rows, with tail rows), lane counts that are not a multiple of 16, the norm
prologue with and without its second addend, determinism, lane-order independence and NaN
propagation.  The error word must stay clear.
"""

import numpy as np
import pytest

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import (Guarded, check_close, dev, gq4_module, host, requires_cuda, tol_bf16,
                            tol_gated, wdev)

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    g = gq4_module()
    g.device_error(clear=True)
    return g


def _diag(got, ref, S):
    """Largest relative error over outputs that do not cancel (|ref| >= 0.1 S)."""
    mask = np.abs(ref) >= 0.1 * S
    if not mask.any():
        return 0.0
    return float((np.abs(got - ref)[mask] / np.abs(ref)[mask]).max())


MATVEC_CASES = [
    # M, K, N, gs
    (16, 4096, 4096, 128),    # the stack's O projection
    (32, 4096, 4096, 128),
    (32, 11008, 4096, 128),   # the stack's down projection (86 groups per column)
    (16, 11008, 4096, 128),
    (16, 32, 1, 32),          # one chunk, one column (too few rows for the tensor-core path)
    (16, 64, 4, 32),          # K inside one partial stage, scale rows in pairs
    (16, 160, 9, 32),         # 5 groups per column: scale rows in fours, one tail row
    (20, 11008, 3, 128),      # 86 groups per column: scale rows in pairs, one tail row
    (17, 96, 7, 96),          # group size that does not divide the 256-code stage
    (31, 288, 130, 32),       # partial last stage, partial tile
    (32, 12800, 19, 256),     # many stages, few columns
    (24, 16384, 300, 1024),   # large groups
    (32, 1024, 1024, 32),     # the single-matvec shape at 32 lanes
]


@pytest.mark.parametrize("M,K,N,gs", MATVEC_CASES)
def test_tc_matvec(gq4, M, K, N, gs):
    w = I.quant_weights(K, N, gs, 1100, M, K, N)
    A = I.activations(M, K, 1100, M, K, N)
    C_ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    out = Guarded((M, N))
    gq4.matvec(dev(A), *wdev(w), gs, C=out.t)
    out.check()
    C = host(out.t)
    check_close(f"tc matvec M{M} K{K} N{N} gs{gs}", C, C_ref, tol_bf16(S))
    # bf16 rounding of both operands: far inside the bound on non-cancelling outputs
    assert _diag(C, C_ref, S) < 2e-2
    assert gq4.device_error() == 0


@pytest.mark.parametrize("M", [16, 32])
def test_tc_quad_stack(gq4, M):
    K, N, gs, n0, n1, n2 = 4096, 6144, 128, 4096, 5120, 6144
    w = I.quant_weights(K, N, gs, 1101, M)
    A = I.activations(M, K, 1101, M)
    outs_ref, sabs = oracle.quad_matvec(A, w.Bq, w.scales, w.zeros, K, N, gs, n0, n1, n2)
    lens = [n0, n1 - n0, n2 - n1, N - n2]
    guards = [Guarded((M, n)) for n in lens]
    gq4.quad_matvec(dev(A), *wdev(w), gs, n0, n1, n2,
                    outs=[g.t if n else None for g, n in zip(guards, lens)])
    for i, (g, n) in enumerate(zip(guards, lens)):
        g.check()
        if n:
            check_close(f"tc quad out{i}", host(g.t), outs_ref[i], tol_bf16(sabs[i]))
    assert gq4.device_error() == 0


@pytest.mark.parametrize("M,K,N,gs,n0,n1,n2", [
    (24, 2560, 10240, 64, 4096, 5120, 6144),   # the quad workload at 24 lanes
    (16, 256, 50, 32, 0, 0, 0),                # everything to out3
    (32, 128, 37, 64, 1, 2, 3),                # single-column segments
])
def test_tc_quad_splits(gq4, M, K, N, gs, n0, n1, n2):
    w = I.quant_weights(K, N, gs, 1102, M, K, N)
    A = I.activations(M, K, 1102, M, K, N)
    outs_ref, sabs = oracle.quad_matvec(A, w.Bq, w.scales, w.zeros, K, N, gs, n0, n1, n2)
    lens = [n0, n1 - n0, n2 - n1, N - n2]
    guards = [Guarded((M, n)) for n in lens]
    gq4.quad_matvec(dev(A), *wdev(w), gs, n0, n1, n2,
                    outs=[g.t if n else None for g, n in zip(guards, lens)])
    for i, (g, n) in enumerate(zip(guards, lens)):
        g.check()
        if n:
            check_close(f"tc quad out{i}", host(g.t), outs_ref[i], tol_bf16(sabs[i]))


@pytest.mark.parametrize("M,K,N,gs,with_b", [
    (16, 4096, 4096, 64, True),     # the norm-prologue workload at 16 lanes
    (32, 4096, 300, 128, False),
    (20, 11008, 64, 128, True),     # the ffn width as K
    (32, 96, 9, 32, True),          # one partial stage
    (32, 480, 130, 96, True),       # 5 groups per column, two tail rows
])
def test_tc_norm(gq4, M, K, N, gs, with_b):
    w = I.quant_weights(K, N, gs, 1103, M, K, N)
    A = I.activations(M, K, 1103, M, K, N)
    A_b = I.activations(M, K, 1104, M, K, N) if with_b else None
    W = I.norm_gain(K, 1103, M, K)
    C_ref, S, res_ref, nout_ref = oracle.norm_matvec(A, A_b, W, 1e-6, w.Bq, w.scales, w.zeros,
                                                     K, N, gs)
    C, res, nout = Guarded((M, N)), Guarded((M, K)), Guarded((M, K))
    gq4.norm_matvec(dev(A), *wdev(w), gs, dev(W), 1e-6, A_b=dev(A_b) if with_b else None,
                    residual_out=res.t, norm_out=nout.t, C=C.t)
    for g in (C, res, nout):
        g.check()
    check_close("tc norm C", host(C.t), C_ref, tol_bf16(S))
    assert np.array_equal(host(res.t).view(np.uint32), res_ref.view(np.uint32)), "residual_out"
    check_close("tc norm_out", host(nout.t), nout_ref, 1e-5 * np.abs(nout_ref) + 1e-7)
    assert gq4.device_error() == 0


@pytest.mark.parametrize("M,K,N,gs,use_norm", [
    (32, 4096, 11008, 128, True),    # the stack's gated call at 32 lanes
    (16, 4096, 11008, 128, False),   # the gated workload at 16 lanes
    (16, 256, 20, 32, False),
    (27, 1024, 130, 64, True),
    (32, 96, 5, 32, True),           # 3 groups per column, one tail row
])
def test_tc_gated(gq4, M, K, N, gs, use_norm):
    wg = I.quant_weights(K, N, gs, 1105, M, K, N, scale_range=I.SCALE_RANGE_GATED)
    wu = I.quant_weights(K, N, gs, 1106, M, K, N, scale_range=I.SCALE_RANGE_GATED)
    A = I.activations(M, K, 1105, M, K, N)
    kw = {}
    if use_norm:
        kw = dict(A_b=I.activations(M, K, 1106, M, K, N), W_norm=I.norm_gain(K, 1105, M, K),
                  eps=1e-6)
    ref = oracle.gated_matvec(A, wg.Bq, wg.scales, wg.zeros, wu.Bq, wu.scales, wu.zeros,
                              K, N, gs, **kw)
    out = Guarded((M, N))
    dkw = {}
    res = nout = None
    if use_norm:
        res, nout = Guarded((M, K)), Guarded((M, K))
        dkw = dict(A_b=dev(kw["A_b"]), W_norm=dev(kw["W_norm"]), eps=1e-6,
                   residual_out=res.t, norm_out=nout.t)
    gq4.gated_matvec(dev(A), *wdev(wg), *wdev(wu), gs, out=out.t, **dkw)
    out.check()
    tol = tol_gated(ref["g"], ref["u"], ref["Sg"], ref["Su"], ref["out"], eps_fn=tol_bf16)
    check_close(f"tc gated M{M} K{K} N{N}", host(out.t), ref["out"], tol)
    if use_norm:
        res.check()
        nout.check()
        assert np.array_equal(host(res.t).view(np.uint32), ref["residual_out"].view(np.uint32))
        check_close("tc gated norm_out", host(nout.t), ref["norm_out"],
                    1e-5 * np.abs(ref["norm_out"]) + 1e-7)
    assert gq4.device_error() == 0


@pytest.mark.parametrize("M", [16, 32])
def test_tc_deterministic_and_lane_order(gq4, M):
    """Same inputs give the same bits; permuting the lanes permutes the outputs
    bit for bit (each lane is one independent column of the MMA)."""
    K, N, gs = 4096, 1000, 128
    w = I.quant_weights(K, N, gs, 1107)
    A = I.activations(M, K, 1107, M)
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    again = host(gq4.matvec(dev(A), *wdev(w), gs))
    assert np.array_equal(C.view(np.uint32), again.view(np.uint32))
    perm = I.rng(1107, M, 1).permutation(M)
    Cp = host(gq4.matvec(dev(np.ascontiguousarray(A[perm])), *wdev(w), gs))
    assert np.array_equal(Cp.view(np.uint32), C[perm].view(np.uint32))


def test_tc_nonfinite_activation_propagates(gq4):
    M, K, N, gs = 16, 512, 40, 32
    w = I.quant_weights(K, N, gs, 1108)
    A = I.activations(M, K, 1108)
    A[3, 17] = np.nan
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    assert np.all(np.isnan(C[3]))
    assert np.all(np.isfinite(np.delete(C, 3, axis=0)))

"""GPU parity of the 2..4-lane kernel (persistent bulk-copy ring, exact fp16
products on the warp-level MMA), against the oracle at the fp32 tolerance.

Covered: plain, quad routing, RMSNorm prologue (with and without A_b),
SiLU-gated gate/up (with and without the norm), dual, both gated inputs;
a single partial tile, one full tile, ragged tiles, fewer columns than SMs,
K not a multiple of 256, group sizes of 128, 256 and 512 (a warp's slice
inside one group), M = 3 (a zero lane in the MMA), the stack's QKV, O and
gate/up calls at M = 4 at full size; lane permutation, repeat calls and
quad == plain bit for bit; a non-finite activation in one lane (that lane's
outputs NaN, the others unchanged); activations over a wide dynamic range.
K split over a cluster (the stack's down projection at M = 4, 2 and 4 chunks,
of unequal sizes, groups of 1 to 4 blocks, fewer columns than clusters) with the
plain, RMSNorm, quad, gated, dual and gated-input forms.
"""

import numpy as np
import pytest
import torch

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import (Guarded, check_close, dev, gq4_module, host, requires_cuda, tol_fp32,
                            tol_gated, wdev)

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    g = gq4_module()
    g.device_error(clear=True)
    yield g
    assert g.device_error() == 0


MATVEC_CASES = [
    # M, K, N, gs
    (2, 128, 1, 128),        # one block, one column
    (2, 256, 16, 128),       # one full tile
    (3, 1152, 17, 128),      # K not a multiple of 256, a ragged second tile
    (4, 4096, 4096, 128),    # the stack's O projection at M = 4
    (2, 4096, 300, 256),     # two blocks per group
    (4, 2048, 33, 512),      # a warp's two blocks inside one group
    (3, 512, 7, 128),        # fewer columns than SMs
    (4, 1024, 152 * 16 + 5, 128),  # every CTA with a ragged range
]


@pytest.mark.parametrize("M,K,N,gs", MATVEC_CASES)
def test_lanes_matvec(gq4, M, K, N, gs):
    w = I.quant_weights(K, N, gs, 1700, M, K, N)
    A = I.activations(M, K, 1700, M, K, N)
    ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    out = Guarded((M, N))
    gq4.matvec(dev(A), *wdev(w), gs, C=out.t)
    out.check()
    check_close(f"lanes matvec M{M} K{K} N{N} gs{gs}", host(out.t), ref, tol_fp32(S))


QUAD_CASES = [
    # M, K, N, gs, n0, n1, n2
    (4, 4096, 6144, 128, 4096, 5120, 6144),   # the stack's QKV call at M = 4
    (3, 1024, 1000, 128, 17, 33, 999),
    (2, 512, 64, 128, 0, 0, 0),               # everything in out3
]


@pytest.mark.parametrize("M,K,N,gs,n0,n1,n2", QUAD_CASES)
def test_lanes_quad(gq4, M, K, N, gs, n0, n1, n2):
    w = I.quant_weights(K, N, gs, 1701, M, K, N)
    A = I.activations(M, K, 1701, M, K, N)
    outs_ref, sabs = oracle.quad_matvec(A, w.Bq, w.scales, w.zeros, K, N, gs, n0, n1, n2)
    lens = [n0, n1 - n0, n2 - n1, N - n2]
    outs = [Guarded((M, n)) for n in lens]
    gq4.quad_matvec(dev(A), *wdev(w), gs, n0, n1, n2, outs=[o.t for o in outs])
    for i, o in enumerate(outs):
        o.check()
        if lens[i]:
            check_close(f"lanes quad out{i}", host(o.t), outs_ref[i], tol_fp32(sabs[i]))
    # the concatenated outputs equal the plain call bit for bit
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    cat = np.concatenate([host(o.t) for o in outs], axis=1)
    assert np.array_equal(cat.view(np.uint32), C.view(np.uint32))


NORM_CASES = [
    # M, K, N, gs, with A_b
    (4, 4096, 4096, 128, True),
    (2, 1024, 70, 256, False),
    (3, 4096, 50, 128, True),
]


@pytest.mark.parametrize("M,K,N,gs,with_b", NORM_CASES)
def test_lanes_norm(gq4, M, K, N, gs, with_b):
    w = I.quant_weights(K, N, gs, 1702, M, K, N)
    A = I.activations(M, K, 1702, M, K, N)
    A_b = I.activations(M, K, 1703, M, K, N) if with_b else None
    W = I.norm_gain(K, 1702, M, K)
    C_ref, S, res_ref, nout_ref = oracle.norm_matvec(A, A_b, W, 1e-6, w.Bq, w.scales, w.zeros, K, N, gs)
    C, res, nout = Guarded((M, N)), Guarded((M, K)), Guarded((M, K))
    gq4.norm_matvec(dev(A), *wdev(w), gs, dev(W), 1e-6, A_b=dev(A_b) if with_b else None,
                    residual_out=res.t, norm_out=nout.t, C=C.t)
    for g in (C, res, nout):
        g.check()
    check_close("lanes norm C", host(C.t), C_ref, tol_fp32(S))
    assert np.array_equal(host(res.t).view(np.uint32), res_ref.view(np.uint32)), "residual_out"
    check_close("lanes norm_out", host(nout.t), nout_ref, 1e-5 * np.abs(nout_ref) + 1e-7)


GATED_CASES = [
    # M, K, N, gs, norm
    (4, 4096, 11008, 128, True),   # the stack's gate/up call at M = 4
    (2, 1024, 37, 128, False),
    (3, 256, 9, 128, True),
]


@pytest.mark.parametrize("M,K,N,gs,use_norm", GATED_CASES)
def test_lanes_gated(gq4, M, K, N, gs, use_norm):
    wg = I.quant_weights(K, N, gs, 1704, M, K, N, scale_range=I.SCALE_RANGE_GATED)
    wu = I.quant_weights(K, N, gs, 1705, M, K, N, scale_range=I.SCALE_RANGE_GATED)
    A = I.activations(M, K, 1704, M, K, N)
    kw = {}
    if use_norm:
        kw = dict(A_b=I.activations(M, K, 1705, M, K, N), W_norm=I.norm_gain(K, 1704, M, K), eps=1e-6)
    ref = oracle.gated_matvec(A, wg.Bq, wg.scales, wg.zeros, wu.Bq, wu.scales, wu.zeros, K, N, gs, **kw)
    out = Guarded((M, N))
    dkw = {}
    res = nout = None
    if use_norm:
        res, nout = Guarded((M, K)), Guarded((M, K))
        dkw = dict(A_b=dev(kw["A_b"]), W_norm=dev(kw["W_norm"]), eps=1e-6, residual_out=res.t,
                   norm_out=nout.t)
    gq4.gated_matvec(dev(A), *wdev(wg), *wdev(wu), gs, out=out.t, **dkw)
    out.check()
    tol = tol_gated(ref["g"], ref["u"], ref["Sg"], ref["Su"], ref["out"])
    check_close(f"lanes gated M{M} N{N}", host(out.t), ref["out"], tol)
    if use_norm:
        res.check()
        nout.check()
        assert np.array_equal(host(res.t).view(np.uint32), ref["residual_out"].view(np.uint32))
        check_close("lanes gated norm_out", host(nout.t), ref["norm_out"],
                    1e-5 * np.abs(ref["norm_out"]) + 1e-7)


@pytest.mark.parametrize("M,K,N,gs", [(4, 1024, 70, 128), (2, 4096, 4096, 128)])
def test_lanes_dual(gq4, M, K, N, gs):
    w0 = I.quant_weights(K, N, gs, 1706, M, K, N, 0)
    w1 = I.quant_weights(K, N, gs, 1706, M, K, N, 1)
    A = I.activations(M, K, 1706, M, K, N)
    C0, C1 = gq4.dual_matvec(dev(A), *wdev(w0), *wdev(w1), gs)
    for name, C, w in (("C0", C0, w0), ("C1", C1, w1)):
        ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
        check_close(f"lanes dual {name}", host(C), ref, tol_fp32(S))
        # each output equals the plain call on its matrix bit for bit
        solo = host(gq4.matvec(dev(A), *wdev(w), gs))
        assert np.array_equal(host(C).view(np.uint32), solo.view(np.uint32)), name


# K split over a cluster: each CTA a chunk of whole groups, rank 0 adds the
# chunks' sums (K past 36 blocks, or more than 32 groups per column)
SPLIT_CASES = [
    # M, K, N, gs
    (4, 11008, 4096, 128),   # the stack's down projection at M = 4 (4 chunks)
    (2, 4736, 37, 128),      # 37 groups: 2 chunks of 18 and 19, ragged tiles
    (3, 8192, 300, 256),     # 2 chunks of 16 groups of two blocks
    (4, 16384, 64, 512),     # 4 chunks of 8 groups of four blocks
    (2, 5120, 5, 128),       # fewer columns than clusters
    (3, 12288, 40, 2048),    # 6 groups of 16 blocks: 3 chunks (4 would leave one empty)
]


@pytest.mark.parametrize("M,K,N,gs", SPLIT_CASES)
def test_lanes_split_matvec(gq4, M, K, N, gs):
    w = I.quant_weights(K, N, gs, 1711, M, K, N)
    A = I.activations(M, K, 1711, M, K, N)
    ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    out = Guarded((M, N))
    gq4.matvec(dev(A), *wdev(w), gs, C=out.t)
    out.check()
    check_close(f"lanes split matvec M{M} K{K} N{N} gs{gs}", host(out.t), ref, tol_fp32(S))
    # repeatable to the bit, and lane m equals a two-lane call on row m
    again = host(gq4.matvec(dev(A), *wdev(w), gs))
    assert np.array_equal(again.view(np.uint32), host(out.t).view(np.uint32))
    pair = host(gq4.matvec(dev(np.ascontiguousarray(A[[M - 1, 0]])), *wdev(w), gs))
    assert np.array_equal(pair[0].view(np.uint32), host(out.t)[M - 1].view(np.uint32))


@pytest.mark.parametrize("M", [2, 4])
def test_lanes_split_norm_quad(gq4, M):
    """RMSNorm prologue (square sums over the chunks) with quad routing, K = 5120 (40 groups)."""
    K, N, gs = 5120, 400, 128
    w = I.quant_weights(K, N, gs, 1712, M, K, N)
    A = I.activations(M, K, 1712, M, K, N)
    A_b = I.activations(M, K, 1713, M, K, N)
    W = I.norm_gain(K, 1712, M, K)
    C_ref, S, res_ref, nout_ref = oracle.norm_matvec(A, A_b, W, 1e-6, w.Bq, w.scales, w.zeros, K, N, gs)
    C, res, nout = Guarded((M, N)), Guarded((M, K)), Guarded((M, K))
    gq4.norm_matvec(dev(A), *wdev(w), gs, dev(W), 1e-6, A_b=dev(A_b), residual_out=res.t,
                    norm_out=nout.t, C=C.t)
    for g in (C, res, nout):
        g.check()
    check_close("lanes split norm C", host(C.t), C_ref, tol_fp32(S))
    assert np.array_equal(host(res.t).view(np.uint32), res_ref.view(np.uint32)), "residual_out"
    check_close("lanes split norm_out", host(nout.t), nout_ref, 1e-5 * np.abs(nout_ref) + 1e-7)
    n0, n1, n2 = 100, 250, 333
    outs_ref, sabs = oracle.quad_matvec(A, w.Bq, w.scales, w.zeros, K, N, gs, n0, n1, n2)
    lens = [n0, n1 - n0, n2 - n1, N - n2]
    outs = [Guarded((M, n)) for n in lens]
    gq4.quad_matvec(dev(A), *wdev(w), gs, n0, n1, n2, outs=[o.t for o in outs])
    for i, o in enumerate(outs):
        o.check()
        check_close(f"lanes split quad out{i}", host(o.t), outs_ref[i], tol_fp32(sabs[i]))


@pytest.mark.parametrize("M,use_norm", [(3, True), (3, False), (2, True)])
def test_lanes_split_gated(gq4, M, use_norm):
    K, N, gs = 5120, 70, 128
    wg = I.quant_weights(K, N, gs, 1714, M, K, N, scale_range=I.SCALE_RANGE_GATED)
    wu = I.quant_weights(K, N, gs, 1715, M, K, N, scale_range=I.SCALE_RANGE_GATED)
    A = I.activations(M, K, 1714, M, K, N)
    kw, dkw = {}, {}
    if use_norm:
        kw = dict(A_b=I.activations(M, K, 1715, M, K, N), W_norm=I.norm_gain(K, 1714, M, K), eps=1e-6)
        dkw = dict(A_b=dev(kw["A_b"]), W_norm=dev(kw["W_norm"]), eps=1e-6)
    ref = oracle.gated_matvec(A, wg.Bq, wg.scales, wg.zeros, wu.Bq, wu.scales, wu.zeros, K, N, gs, **kw)
    out = Guarded((M, N))
    gq4.gated_matvec(dev(A), *wdev(wg), *wdev(wu), gs, out=out.t, **dkw)
    out.check()
    tol = tol_gated(ref["g"], ref["u"], ref["Sg"], ref["Su"], ref["out"])
    check_close(f"lanes split gated M{M} norm={use_norm}", host(out.t), ref["out"], tol)


def test_lanes_split_dual_and_gated_input(gq4):
    M, K, N, gs = 4, 6144, 90, 128
    w0 = I.quant_weights(K, N, gs, 1716, M, K, N, 0)
    w1 = I.quant_weights(K, N, gs, 1716, M, K, N, 1)
    A = I.activations(M, K, 1716, M, K, N)
    C0, C1 = gq4.dual_matvec(dev(A), *wdev(w0), *wdev(w1), gs)
    for name, C, w in (("C0", C0, w0), ("C1", C1, w1)):
        ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
        check_close(f"lanes split dual {name}", host(C), ref, tol_fp32(S))
    G = I.activations(M, K, 1717, M, K, N)
    C = host(gq4.swiglu_gated_matvec(dev(A), dev(G), *wdev(w0), gs))
    ref, S, _ = oracle.gated_input_matvec("swiglu", A, G, w0.Bq, w0.scales, w0.zeros, K, N, gs)
    check_close("lanes split gated input", C, ref, tol_fp32(S))


@pytest.mark.parametrize("kind", ["sigmoid", "swiglu"])
def test_lanes_gated_input(gq4, kind):
    M, K, N, gs = 3, 2048, 100, 128
    w = I.quant_weights(K, N, gs, 1707)
    X = I.activations(M, K, 1707, 0)
    G = I.activations(M, K, 1707, 1)
    fn = gq4.sigmoid_gated_matvec if kind == "sigmoid" else gq4.swiglu_gated_matvec
    C = host(fn(dev(X), dev(G), *wdev(w), gs))
    ref, S, _ = oracle.gated_input_matvec(kind, X, G, w.Bq, w.scales, w.zeros, K, N, gs)
    check_close(f"lanes gated input {kind}", C, ref, tol_fp32(S))


def test_lanes_permutation_and_repeat(gq4):
    """Permuting the lanes permutes the outputs; a repeated call gives the same bits."""
    M, K, N, gs = 4, 4096, 200, 128
    w = I.quant_weights(K, N, gs, 1708)
    A = I.activations(M, K, 1708)
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    again = host(gq4.matvec(dev(A), *wdev(w), gs))
    assert np.array_equal(C.view(np.uint32), again.view(np.uint32))
    perm = [2, 0, 3, 1]
    Cp = host(gq4.matvec(dev(A[perm]), *wdev(w), gs))
    assert np.array_equal(Cp.view(np.uint32), C[perm].view(np.uint32))
    # three lanes: the same bits as the first three rows of the four-lane call
    C3 = host(gq4.matvec(dev(A[:3]), *wdev(w), gs))
    assert np.array_equal(C3.view(np.uint32), C[:3].view(np.uint32))


def test_lanes_nonfinite_lane(gq4):
    """inf, -inf or NaN in one lane's activations makes that lane's outputs NaN only."""
    M, K, N, gs = 4, 1024, 40, 128
    w = I.quant_weights(K, N, gs, 1709)
    A = I.activations(M, K, 1709)
    base = host(gq4.matvec(dev(A), *wdev(w), gs))
    for lane, val in ((1, np.inf), (2, -np.inf), (3, np.nan)):
        B = A.copy()
        B[lane, 777] = val
        C = host(gq4.matvec(dev(B), *wdev(w), gs))
        assert np.all(np.isnan(C[lane])), (lane, val)
        others = [m for m in range(M) if m != lane]
        assert np.array_equal(C[others].view(np.uint32), base[others].view(np.uint32)), (lane, val)


def test_lanes_dynamic_range(gq4):
    """Outliers 100x and 1000x inside blocks, and whole lanes scaled by 1e-30 and 1e20."""
    M, K, N, gs = 4, 2048, 64, 128
    w = I.quant_weights(K, N, gs, 1710)
    A = I.activations(M, K, 1710).astype(np.float64)
    A[0, ::97] *= 100.0
    A[1, 5::131] *= 1000.0
    A[2] *= 1e-30
    A[3] *= 1e20
    A = A.astype(np.float32)
    ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    check_close("lanes dynamic range", C, ref, tol_fp32(S))

"""GPU parity: every entry point against the oracle, element by element.

Cases span several column tiles and a ragged tail, the five workloads at
their full sizes (sampled columns where the oracle would take too long), the
edge cases of the method (N = 1, K = group size, empty quad segments, split
points at 0 and N, odd lane counts), and lanes M in 1..32.
"""

import numpy as np
import pytest

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import (Guarded, check_close, dev, gq4_module, host, requires_cuda, tol_bf16,
                            tol_fp32, tol_gated, wdev)

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    return gq4_module()


def _tol_for(M):
    """16..32 lanes run on the bf16 tensor-core kernel, fewer in f32."""
    return tol_bf16 if M >= 16 else tol_fp32


# ---------------------------------------------------------------------------
# plain matvec
# ---------------------------------------------------------------------------

MATVEC_CASES = [
    # M, K, N, gs
    (1, 1024, 1024, 32),     # the single-matvec workload
    (1, 32, 1, 32),          # smallest: one chunk, one column
    (1, 64, 17, 64),         # K = gs, ragged column tile
    (2, 256, 33, 32),
    (3, 512, 100, 128),
    (4, 2560, 257, 64),
    (5, 1024, 40, 32),
    (8, 4096, 31, 128),
    (16, 1024, 64, 64),
    (32, 512, 48, 32),
    (1, 11008, 37, 128),     # 86 groups per column (8-byte aligned scale rows)
    (1, 12800, 19, 256),     # two K tiles of staged activations at M=1
    (7, 4096, 23, 64),       # several K tiles at M>4
    (1, 65536, 9, 128),      # K past the one-lane kernel's shared-memory plan (general kernel)
]


@pytest.mark.parametrize("M,K,N,gs", MATVEC_CASES)
def test_matvec(gq4, M, K, N, gs):
    w = I.quant_weights(K, N, gs, 900, M, K, N)
    A = I.activations(M, K, 900, M, K, N)
    C_ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    out = Guarded((M, N))
    gq4.matvec(dev(A), *wdev(w), gs, C=out.t)
    out.check()
    check_close(f"matvec M{M} K{K} N{N} gs{gs}", host(out.t), C_ref, _tol_for(M)(S))


# ---------------------------------------------------------------------------
# quad-output routing
# ---------------------------------------------------------------------------

QUAD_CASES = [
    # M, K, N, gs, n0, n1, n2
    (1, 2560, 10240, 64, 4096, 5120, 6144),   # the quad QKV workload
    (1, 256, 50, 32, 16, 24, 40),
    (2, 256, 50, 32, 0, 0, 0),                 # everything to out3
    (1, 256, 50, 32, 50, 50, 50),              # everything to out0
    (3, 128, 37, 64, 1, 2, 3),                 # single-column segments
    (4, 512, 64, 128, 0, 32, 32),              # empty out0 and out2
    (1, 4096, 6144, 128, 4096, 5120, 6144),    # the stack's qkv (out3 empty)
]


@pytest.mark.parametrize("M,K,N,gs,n0,n1,n2", QUAD_CASES)
def test_quad(gq4, M, K, N, gs, n0, n1, n2):
    w = I.quant_weights(K, N, gs, 901, M, K, N)
    A = I.activations(M, K, 901, M, K, N)
    outs_ref, sabs = oracle.quad_matvec(A, w.Bq, w.scales, w.zeros, K, N, gs, n0, n1, n2)
    lens = [n0, n1 - n0, n2 - n1, N - n2]
    guards = [Guarded((M, n)) for n in lens]
    outs = [g.t if n else None for g, n in zip(guards, lens)]
    gq4.quad_matvec(dev(A), *wdev(w), gs, n0, n1, n2, outs=outs)
    for i, (g, n) in enumerate(zip(guards, lens)):
        g.check()
        if n:
            check_close(f"quad out{i}", host(g.t), outs_ref[i], _tol_for(M)(sabs[i]))


# ---------------------------------------------------------------------------
# norm prologue
# ---------------------------------------------------------------------------

NORM_CASES = [
    # M, K, N, gs, with A_b
    (1, 4096, 4096, 64, True),                 # the norm-prologue workload
    (1, 256, 19, 32, False),
    (3, 1024, 40, 128, True),
    (8, 4096, 33, 64, True),                   # K tiles at M=8
    (4, 4096, 50, 128, True),                  # stack hidden size at M=4 (largest K tile)
    (2, 11008, 30, 128, True),                 # ffn size at M=2 (largest K tile)
    (32, 512, 20, 32, True),
    (1, 12800, 40, 256, True),                 # one lane, K past one prologue batch
]


@pytest.mark.parametrize("M,K,N,gs,with_b", NORM_CASES)
def test_norm_matvec(gq4, M, K, N, gs, with_b):
    w = I.quant_weights(K, N, gs, 902, M, K, N)
    A = I.activations(M, K, 902, M, K, N)
    A_b = I.activations(M, K, 903, M, K, N) if with_b else None
    W = I.norm_gain(K, 902, M, K)
    C_ref, S, res_ref, nout_ref = oracle.norm_matvec(A, A_b, W, 1e-6, w.Bq, w.scales, w.zeros,
                                                     K, N, gs)
    C = Guarded((M, N))
    res = Guarded((M, K))
    nout = Guarded((M, K))
    gq4.norm_matvec(dev(A), *wdev(w), gs, dev(W), 1e-6, A_b=dev(A_b) if with_b else None,
                    residual_out=res.t, norm_out=nout.t, C=C.t)
    for g in (C, res, nout):
        g.check()
    check_close("norm C", host(C.t), C_ref, _tol_for(M)(S))
    assert np.array_equal(host(res.t).view(np.uint32), res_ref.view(np.uint32)), "residual_out"
    check_close("norm_out", host(nout.t), nout_ref, 1e-5 * np.abs(nout_ref) + 1e-7)


def test_norm_without_side_outputs(gq4):
    M, K, N, gs = 2, 1024, 48, 64
    w = I.quant_weights(K, N, gs, 904)
    A = I.activations(M, K, 904)
    A_b = I.activations(M, K, 905)
    W = I.norm_gain(K, 904)
    C_ref, S, _, _ = oracle.norm_matvec(A, A_b, W, 1e-6, w.Bq, w.scales, w.zeros, K, N, gs)
    C = gq4.norm_matvec(dev(A), *wdev(w), gs, dev(W), 1e-6, A_b=dev(A_b))
    check_close("norm C (no side outputs)", host(C), C_ref, tol_fp32(S))


# ---------------------------------------------------------------------------
# SiLU-gated gate/up
# ---------------------------------------------------------------------------

GATED_CASES = [
    # M, K, N, gs, norm
    (1, 4096, 11008, 128, False),              # the gated workload
    (1, 4096, 11008, 128, True),               # with the norm prologue (stack form)
    (1, 256, 21, 32, False),
    (4, 1024, 70, 64, True),
    (4, 4096, 300, 128, True),                 # the stack's gated call at M=4
    (16, 512, 24, 128, False),
    (32, 256, 20, 32, True),
]


@pytest.mark.parametrize("M,K,N,gs,use_norm", GATED_CASES)
def test_gated(gq4, M, K, N, gs, use_norm):
    wg = I.quant_weights(K, N, gs, 906, M, K, N, scale_range=I.SCALE_RANGE_GATED)
    wu = I.quant_weights(K, N, gs, 907, M, K, N, scale_range=I.SCALE_RANGE_GATED)
    A = I.activations(M, K, 906, M, K, N)
    kw = {}
    if use_norm:
        A_b = I.activations(M, K, 907, M, K, N)
        W = I.norm_gain(K, 906, M, K)
        kw = dict(A_b=A_b, W_norm=W, eps=1e-6)
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
    tol = tol_gated(ref["g"], ref["u"], ref["Sg"], ref["Su"], ref["out"], eps_fn=_tol_for(M))
    check_close(f"gated M{M} K{K} N{N}", host(out.t), ref["out"], tol)
    if use_norm:
        res.check()
        nout.check()
        assert np.array_equal(host(res.t).view(np.uint32), ref["residual_out"].view(np.uint32))
        check_close("gated norm_out", host(nout.t), ref["norm_out"],
                    1e-5 * np.abs(ref["norm_out"]) + 1e-7)

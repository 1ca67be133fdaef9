"""GPU test of back-to-back dependent calls through the single-call entry points.

Calls with M = 1 and 16 <= M <= 32 are launched with programmatic dependent
launch: a call's CTAs may start, and stream their weights, while the
previous call on the stream is still running, and must wait for it before
reading activations.  Each chain below enqueues every call before a single
synchronisation; every intermediate has a buffer of its own, filled with NaN
first, and each call is checked against the oracle on the inputs the GPU
produced for it, so a call that read its activations early fails.
"""

import numpy as np
import pytest
import torch

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import check_close, dev, gq4_module, host, requires_cuda, tol_bf16, tol_fp32, tol_gated, wdev

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    g = gq4_module()
    g.device_error(clear=True)
    return g


@pytest.mark.parametrize("M", [1, 16])
def test_chain_of_matvecs(gq4, M):
    """24 chained matvecs h_{i+1} = W_i h_i (K = N = 1024, group 64), one sync at the end."""
    K, gs = 1024, 64
    h = dev(I.activations(M, K, 1400, M))
    chain = []
    for i in range(24):
        w = I.quant_weights(K, K, gs, 1400, M, i, scale_range=(0.001, 0.004))
        C = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
        gq4.matvec(h, *wdev(w), gs, C=C)
        chain.append((h, w, C))
        h = C
    torch.cuda.synchronize()
    tol = tol_fp32 if M == 1 else tol_bf16
    for i, (A, w, C) in enumerate(chain):
        ref, S = oracle.matvec(host(A), w.Bq, w.scales, w.zeros, K, K, gs)
        check_close(f"link {i}", host(C), ref, tol(S))
    assert gq4.device_error() == 0


def test_chain_of_mixed_layer_calls(gq4):
    """Three small decode layers (quad, O, gated with its norm prologue reading O, down),
    M = 1, 12 calls enqueued back to back."""
    H, F, gs = 512, 1344, 32
    QKV = (512, 128, 128)
    n0, n1, n2 = QKV[0], QKV[0] + QKV[1], sum(QKV)
    h = dev(I.activations(1, H, 1401, 0))
    nan = lambda n: torch.full((1, n), float("nan"), dtype=torch.float32, device="cuda")
    layers = []
    for li in range(3):
        wqkv = I.quant_weights(H, n2, gs, 1401, li, 1)
        wo = I.quant_weights(H, H, gs, 1401, li, 2)
        wg = I.quant_weights(H, F, gs, 1401, li, 3, scale_range=I.SCALE_RANGE_GATED)
        wu = I.quant_weights(H, F, gs, 1401, li, 4, scale_range=I.SCALE_RANGE_GATED)
        wd = I.quant_weights(F, H, gs, 1401, li, 5)
        W = dev(I.norm_gain(H, 1401, li))
        q, k, v, o, res, f, hn = nan(QKV[0]), nan(QKV[1]), nan(QKV[2]), nan(H), nan(H), nan(F), nan(H)
        gq4.quad_matvec(h, *wdev(wqkv), gs, n0, n1, n2, outs=[q, k, v, None])
        gq4.matvec(q, *wdev(wo), gs, C=o)
        gq4.gated_matvec(h, *wdev(wg), *wdev(wu), gs, W_norm=W, A_b=o, residual_out=res, out=f)
        gq4.matvec(f, *wdev(wd), gs, C=hn)
        layers.append((h, wqkv, q, k, v, wo, o, wg, wu, W, res, f, wd, hn))
        h = hn
    torch.cuda.synchronize()
    for li, (h, wqkv, q, k, v, wo, o, wg, wu, W, res, f, wd, hn) in enumerate(layers):
        outs, sabs = oracle.quad_matvec(host(h), wqkv.Bq, wqkv.scales, wqkv.zeros, H, n2, gs, n0, n1, n2)
        for i, t in enumerate((q, k, v)):
            check_close(f"layer {li} qkv{i}", host(t), outs[i], tol_fp32(sabs[i]))
        C, S = oracle.matvec(host(q), wo.Bq, wo.scales, wo.zeros, H, H, gs)
        check_close(f"layer {li} o", host(o), C, tol_fp32(S))
        r = oracle.gated_matvec(host(h), wg.Bq, wg.scales, wg.zeros, wu.Bq, wu.scales, wu.zeros, H, F, gs,
                                A_b=host(o), W_norm=host(W), eps=1e-6)
        check_close(f"layer {li} gated", host(f), r["out"], tol_gated(r["g"], r["u"], r["Sg"], r["Su"], r["out"]))
        assert np.array_equal(host(res).view(np.uint32), r["residual_out"].view(np.uint32))
        C, S = oracle.matvec(host(f), wd.Bq, wd.scales, wd.zeros, F, H, gs)
        check_close(f"layer {li} down", host(hn), C, tol_fp32(S))
    assert gq4.device_error() == 0

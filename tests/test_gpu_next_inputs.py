"""GPU parity of the dual projection and the gated-input matvecs.

* gq4_dual_matvec (DualMatVecInt4): each output against the oracle matvec of
  its matrix; at M = 1 bit for bit equal to gq4_matvec of each matrix.
* gq4_sigmoid_gated_matvec (GatedMatVecInt4: X * sigmoid(G)) and
  gq4_swiglu_gated_matvec (SwiGLUGatedMatVecInt4: silu(G) * X): against the
  oracle's gated-input matvec, and a saturated gate against the plain matvec.
One lane runs on the streaming kernel, more lanes on the CUDA-core kernel.
"""

import numpy as np
import pytest
import torch

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import check_close, dev, gq4_module, host, requires_cuda, tol_fp32, wdev

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    g = gq4_module()
    g.device_error(clear=True)
    return g


DUAL_CASES = [
    # M, K, N, gs
    (1, 4096, 4096, 128),     # q_proj + gate_proj shaped pair
    (1, 2560, 1001, 64),      # ragged columns
    (1, 11008, 77, 128),      # long columns
    (3, 1024, 40, 32),
    (16, 512, 33, 64),
    (32, 256, 20, 32),
]


@pytest.mark.parametrize("M,K,N,gs", DUAL_CASES)
def test_dual(gq4, M, K, N, gs):
    w0 = I.quant_weights(K, N, gs, 1500, M, K, N, 0)
    w1 = I.quant_weights(K, N, gs, 1500, M, K, N, 1)
    A = I.activations(M, K, 1500, M, K, N)
    C0, C1 = gq4.dual_matvec(dev(A), *wdev(w0), *wdev(w1), gs)
    torch.cuda.synchronize()
    for name, C, w in (("C0", C0, w0), ("C1", C1, w1)):
        ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
        check_close(f"dual {name}", host(C), ref, tol_fp32(S))
    if M == 1:
        for C, w in ((C0, w0), (C1, w1)):
            solo = host(gq4.matvec(dev(A), *wdev(w), gs))
            assert np.array_equal(host(C).view(np.uint32), solo.view(np.uint32))
    assert gq4.device_error() == 0


GATED_INPUT_CASES = [
    # M, K, N, gs
    (1, 4096, 4096, 128),     # o_proj shaped
    (1, 4096, 2048, 64),
    (1, 12800, 33, 256),      # K past one prologue batch
    (4, 1024, 70, 32),
    (16, 512, 24, 128),
]


@pytest.mark.parametrize("kind", ["sigmoid", "swiglu"])
@pytest.mark.parametrize("M,K,N,gs", GATED_INPUT_CASES)
def test_gated_input(gq4, kind, M, K, N, gs):
    w = I.quant_weights(K, N, gs, 1501, M, K, N)
    X = I.activations(M, K, 1501, M, K, N, 0)
    G = I.activations(M, K, 1501, M, K, N, 1)
    fn = gq4.sigmoid_gated_matvec if kind == "sigmoid" else gq4.swiglu_gated_matvec
    C = host(fn(dev(X), dev(G), *wdev(w), gs))
    ref, S, _ = oracle.gated_input_matvec(kind, X, G, w.Bq, w.scales, w.zeros, K, N, gs)
    check_close(f"{kind} M={M}", C, ref, tol_fp32(S))
    assert gq4.device_error() == 0


@pytest.mark.parametrize("M", [1, 4])
def test_saturated_gate(gq4, M):
    """A gate of 64: sigmoid passes X (the plain matvec), silu scales it by 64."""
    K, N, gs = 4096, 300, 128
    w = I.quant_weights(K, N, gs, 1502, M)
    X = I.activations(M, K, 1502, M)
    G = np.full((M, K), 64.0, np.float32)
    ref, S = oracle.matvec(X, w.Bq, w.scales, w.zeros, K, N, gs)
    C = host(gq4.sigmoid_gated_matvec(dev(X), dev(G), *wdev(w), gs))
    check_close("sigmoid(64)", C, ref, tol_fp32(S))
    C = host(gq4.swiglu_gated_matvec(dev(X), dev(G), *wdev(w), gs))
    check_close("silu(64)", C, 64.0 * ref, tol_fp32(64.0 * S))
    assert gq4.device_error() == 0


@pytest.mark.parametrize("kind", ["sigmoid", "swiglu"])
@pytest.mark.parametrize("M", [1, 4])
def test_wide_gate(gq4, kind, M):
    """Gates spread over +-100: e^-g overflows (the gate is exactly 0) or
    vanishes (sigmoid 1, silu g) for many of them; against the oracle."""
    K, N, gs = 4096, 257, 128
    w = I.quant_weights(K, N, gs, 1503, M)
    X = I.activations(M, K, 1503, M, 0)
    G = (40.0 * I.activations(M, K, 1503, M, 1)).clip(-100.0, 100.0).astype(np.float32)
    fn = gq4.sigmoid_gated_matvec if kind == "sigmoid" else gq4.swiglu_gated_matvec
    C = host(fn(dev(X), dev(G), *wdev(w), gs))
    ref, S, _ = oracle.gated_input_matvec(kind, X, G, w.Bq, w.scales, w.zeros, K, N, gs)
    check_close(f"wide {kind} M={M}", C, ref, tol_fp32(S))
    assert gq4.device_error() == 0

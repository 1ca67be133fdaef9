"""GPU parity of the int4 GEMM for prefill and wide batches (gq4_gemm).

Rows run in chunks of up to 32 on the bf16 tensor-core kernel (fewer than 16
padded to 16), so every row is held to the bf16 tolerance against the
oracle's double matvec.  Cases cover a single chunk smaller than 16 rows,
ragged tails of 1 and 15 rows, several whole chunks, ragged columns and
group sizes 32 to 128; a 512 x 4096 x 4096 product is checked on sampled
columns; a whole 32-row chunk equals gq4_matvec of those rows bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import check_close, dev, gq4_module, host, requires_cuda, tol_bf16, wdev

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    g = gq4_module()
    g.device_error(clear=True)
    return g


GEMM_CASES = [
    # M, K, N, gs
    (1, 2048, 100, 64),
    (7, 4096, 300, 64),       # one chunk of 7 rows, padded to 16
    (33, 1024, 200, 64),      # a whole chunk and a 1-row tail
    (47, 512, 130, 32),       # a 15-row tail
    (64, 4096, 257, 128),
    (100, 2048, 96, 128),
    (256, 4096, 512, 128),
]


@pytest.mark.parametrize("M,K,N,gs", GEMM_CASES)
def test_gemm(gq4, M, K, N, gs):
    w = I.quant_weights(K, N, gs, 1900, M, K, N)
    A = I.activations(M, K, 1900, M, K, N)
    C = host(gq4.gemm(dev(A), *wdev(w), gs))
    ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    check_close(f"gemm M={M}", C, ref, tol_bf16(S))
    assert gq4.device_error() == 0


def test_gemm_chunk_equals_matvec(gq4):
    """Rows 32..63 of a GEMM are the 32-lane matvec of those rows, bit for bit."""
    M, K, N, gs = 80, 2048, 300, 128
    w = I.quant_weights(K, N, gs, 1901)
    A = I.activations(M, K, 1901)
    C = host(gq4.gemm(dev(A), *wdev(w), gs))
    C32 = host(gq4.matvec(dev(np.ascontiguousarray(A[32:64])), *wdev(w), gs))
    assert np.array_equal(C[32:64].view(np.uint32), C32.view(np.uint32))


def test_gemm_prefill_sampled(gq4):
    """512 prompt rows through a 4096 x 4096 projection (gs 128): 48 sampled
    columns, including the first and the last, against the oracle."""
    M, K, N, gs = 512, 4096, 4096, 128
    w = I.quant_weights(K, N, gs, 1902)
    A = I.activations(M, K, 1902)
    C = host(gq4.gemm(dev(A), *wdev(w), gs))
    cols = np.unique(np.concatenate([[0, N - 1], I.rng(1902, 9).integers(0, N, 46)])).astype(np.int32)
    ref, S = oracle.dot_cols(A.astype(np.float64), w.Bq, w.scales, w.zeros, K, gs, cols)
    check_close("gemm 512x4096x4096", C[:, cols], ref, tol_bf16(S))
    assert np.all(np.isfinite(C))

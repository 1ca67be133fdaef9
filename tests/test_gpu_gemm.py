"""GPU parity of the int4 GEMM for prefill and wide batches (gq4_gemm).

Every row runs on the bf16 tensor cores and is held to the bf16 tolerance
against the oracle's double matvec.  With a workspace and more than 32 rows
the dedicated GEMM kernel runs (tiles of 128 columns by 64, 128 or 256
rows); without one, rows run in chunks of up to 32 on the decode kernel.
Cases cover ragged rows and columns, group sizes 32 to 128, scale rows that
need the tail copies (K / gs = 3, so 4-row super-rows, and N not a multiple
of 4), sampled 512- and 2048-row products of a 4096 x 4096 projection, and
agreement of the two paths; a 32-row chunk equals gq4_matvec bit for bit.
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
    (7, 4096, 300, 64),       # M <= 32: one chunk of 7 rows, padded to 16
    (33, 1024, 200, 64),      # GEMM kernel: one 64-row tile, 31 rows past M
    (47, 512, 130, 32),
    (40, 384, 130, 128),      # K / gs = 3: scale super-rows of 4, 2 tail rows
    (64, 4096, 257, 128),
    (100, 2048, 96, 128),
    (256, 4096, 512, 128),
    (300, 1024, 1000, 32),
]


@pytest.mark.parametrize("chunked", [False, True])
@pytest.mark.parametrize("M,K,N,gs", GEMM_CASES)
def test_gemm(gq4, M, K, N, gs, chunked):
    w = I.quant_weights(K, N, gs, 1900, M, K, N)
    A = I.activations(M, K, 1900, M, K, N)
    C = host(gq4.gemm(dev(A), *wdev(w), gs, workspace=False if chunked else None))
    ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    check_close(f"gemm M={M} chunked={chunked}", C, ref, tol_bf16(S))
    assert gq4.device_error() == 0


def test_gemm_chunk_equals_matvec(gq4):
    """Rows 32..63 of a GEMM are the 32-lane matvec of those rows, bit for bit."""
    M, K, N, gs = 80, 2048, 300, 128
    w = I.quant_weights(K, N, gs, 1901)
    A = I.activations(M, K, 1901)
    C = host(gq4.gemm(dev(A), *wdev(w), gs, workspace=False))
    C32 = host(gq4.matvec(dev(np.ascontiguousarray(A[32:64])), *wdev(w), gs))
    assert np.array_equal(C[32:64].view(np.uint32), C32.view(np.uint32))


@pytest.mark.parametrize("M", [512, 2048])
def test_gemm_prefill_sampled(gq4, M):
    """512 and 2048 prompt rows through a 4096 x 4096 projection (gs 128): 48
    sampled columns, including the first and the last, against the oracle;
    every output finite."""
    K, N, gs = 4096, 4096, 128
    w = I.quant_weights(K, N, gs, 1902)
    A = I.activations(M, K, 1902, M)
    C = host(gq4.gemm(dev(A), *wdev(w), gs))
    cols = np.unique(np.concatenate([[0, N - 1], I.rng(1902, 9).integers(0, N, 46)])).astype(np.int32)
    ref, S = oracle.dot_cols(A.astype(np.float64), w.Bq, w.scales, w.zeros, K, gs, cols)
    check_close(f"gemm {M}x4096x4096", C[:, cols], ref, tol_bf16(S))
    assert np.all(np.isfinite(C))
    assert gq4.device_error() == 0


def test_gemm_paths_agree(gq4):
    """The GEMM kernel and the 32-row chunks differ only by f32 summation order:
    within twice the bf16 bound of each other on the same products."""
    M, K, N, gs = 200, 2048, 384, 64
    w = I.quant_weights(K, N, gs, 1903)
    A = I.activations(M, K, 1903)
    C1 = host(gq4.gemm(dev(A), *wdev(w), gs))
    C2 = host(gq4.gemm(dev(A), *wdev(w), gs, workspace=False))
    _, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    check_close("GEMM kernel vs chunks", C1, C2, 2 * tol_bf16(S))

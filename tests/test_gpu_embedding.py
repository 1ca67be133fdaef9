"""GPU parity of the int4 embedding gather (gq4_embedding).

Each output is fl(fl(q - zero) * scale) of one table row, the same binary32
operations as the oracle, so the bar is bit equality.  Cases: a single
decode token, ragged widths (segments of 1024 elements cut short), group
sizes 32 to 160, repeated ids, ids outside the table (NaN rows and device
error bit 4), T = 0, and an 8192-token gather from a 32000 x 4096 table
compared in full.
"""

import numpy as np
import pytest
import torch

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import dev, gq4_module, host, requires_cuda, wdev

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    g = gq4_module()
    g.device_error(clear=True)
    return g


def token_ids(T, V, *tags):
    return I.rng(*tags).integers(0, V, size=T, dtype=np.int32)


def check_rows(out, ref):
    out = np.asarray(out)
    assert np.array_equal(np.isnan(out), np.isnan(ref))
    ok = np.isnan(ref) | (out.view(np.uint32) == ref.view(np.uint32))
    assert ok.all(), f"{int((~ok).sum())} elements differ"


EMBED_CASES = [
    # T, K, V, gs
    (1, 4096, 32000, 128),    # one decode token
    (7, 2560, 1000, 64),      # 640 float4 per row: segments of 256, 256, 128
    (33, 384, 77, 96),        # one short segment, a group size that is not a power of two
    (300, 4096, 5000, 32),
    (5, 1280, 11, 160),
    (64, 11008, 40, 128),
]


@pytest.mark.parametrize("T,K,V,gs", EMBED_CASES)
def test_embedding(gq4, T, K, V, gs):
    w = I.quant_weights(K, V, gs, 1800, T, K, V)
    ids = token_ids(T, V, 1800, T, K, V)
    out = gq4.embedding(dev(ids), *wdev(w), gs)
    torch.cuda.synchronize()
    ref, bad = oracle.embedding(ids, w.Bq, w.scales, w.zeros, K, gs)
    assert bad == 0
    check_rows(host(out), ref)
    assert gq4.device_error() == 0


def test_embedding_repeated_and_bad_ids(gq4):
    K, V, gs = 2048, 300, 128
    w = I.quant_weights(K, V, gs, 1801)
    ids = np.array([0, 299, 5, 5, -1, 300, 2**31 - 1, -2**31, 17, 0], np.int32)
    gq4.device_error(clear=True)
    out = gq4.embedding(dev(ids), *wdev(w), gs)
    torch.cuda.synchronize()
    ref, bad = oracle.embedding(ids, w.Bq, w.scales, w.zeros, K, gs)
    assert bad == 4
    check_rows(host(out), ref)
    assert gq4.device_error(clear=True) == 1 << 4
    out = gq4.embedding(dev(ids[:4]), *wdev(w), gs)
    torch.cuda.synchronize()
    assert gq4.device_error() == 0


def test_embedding_empty(gq4):
    K, V, gs = 256, 10, 32
    w = I.quant_weights(K, V, gs, 1802)
    out = gq4.embedding(torch.empty(0, dtype=torch.int32, device="cuda"), *wdev(w), gs)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, K)


def test_embedding_prefill_full(gq4):
    """8192 tokens from a 32000 x 4096 table (gs 128), every element compared."""
    T, K, V, gs = 8192, 4096, 32000, 128
    w = I.quant_weights(K, V, gs, 1803)
    ids = token_ids(T, V, 1803)
    out = gq4.embedding(dev(ids), *wdev(w), gs)
    torch.cuda.synchronize()
    ref, bad = oracle.embedding(ids, w.Bq, w.scales, w.zeros, K, gs)
    assert bad == 0
    check_rows(host(out), ref)

"""GPU integer unpack and binary32 dequant: bit-exact against the oracle.

Both test kernels go through the same in-register extraction as the matvec
kernels (mask in place, OR in the exponent of 2^23, subtract), so these tests
pin that extraction code on the device.
"""

import numpy as np
import pytest

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import dev, gq4_module, host, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]

EDGE_WORDS = [0x00000000, 0xFFFFFFFF, 0x76543210, 0xFEDCBA98, 0x0F0F0F0F, 0xF0F0F0F0,
              0x80000000, 0x00000001, 0x12345678, 0x89ABCDEF]


@pytest.fixture(scope="module")
def gq4():
    return gq4_module()


@pytest.mark.parametrize("K,N", [(32, 1), (1024, 1024), (11008, 5), (64, 1000)])
def test_unpack_random(gq4, K, N):
    Bq = I.words_u32((N, K // 8), 950, K, N)
    got = host(gq4.unpack(dev(Bq), K))
    assert np.array_equal(got, oracle.unpack(Bq, K, N))


def test_unpack_edge_words(gq4):
    words = np.array(EDGE_WORDS * 4, np.uint32)[:32].reshape(1, 32)  # one column, K = 256
    K = 256
    got = host(gq4.unpack(dev(words), K))
    assert np.array_equal(got, oracle.unpack(words, K, 1))
    # and the fixed words read as their codes
    assert list(got[0, 16:24]) == list(range(8))       # 0x76543210 is word 2
    assert list(got[0, 24:32]) == list(range(8, 16))   # 0xFEDCBA98 is word 3


@pytest.mark.parametrize("K,N,gs", [(1024, 1024, 32), (4096, 7, 128), (256, 33, 64)])
def test_dequant_bit_exact(gq4, K, N, gs):
    w = I.quant_weights(K, N, gs, 951, K, N)
    got = host(gq4.dequant(dev(w.Bq), dev(w.scales), dev(w.zeros), K, gs))
    ref = oracle.dequant_f32(w.Bq, w.scales, w.zeros, K, N, gs)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_extreme_zeros(gq4):
    """Zero points outside 0..15, negative, tiny and large stay exact in the extraction."""
    K, N, gs = 256, 6, 32
    G = K // gs
    Bq = I.words_u32((N, K // 8), 952)
    zeros = np.array([[-3.5, 0.0, 15.0, 7.999999, 1e-7, -1e6, 100.25, 2.0 ** 20]] * N,
                     np.float32)[:, :G]
    scales = I.uniform_f32((N, G), 0.001, 3.0, 952)
    got = host(gq4.dequant(dev(Bq), dev(scales), dev(zeros), K, gs))
    ref = oracle.dequant_f32(Bq, scales, zeros, K, N, gs)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))

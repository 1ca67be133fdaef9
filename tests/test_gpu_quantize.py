"""GPU parity of the format producers: gq4_quantize and gq4_from_mlx.

Both decide integers (codes) and single binary32 values (scale, zero) with
the same one-rounding-per-step operations as the oracle, so the bar is bit
equality: Bq word for word, scales and zeros value for value (NaN where the
oracle has NaN).  Shapes cover narrow groups (several per warp, a group size
of 96 that does not divide a warp), wide groups (more than 32 words, two
passes), ragged column counts, and the 4096 x 11008 gate/up projection in
full.  Round trips check the codes through the library's dequant and matvec.
"""

import numpy as np
import pytest
import torch

import oracle
from int4_group_quantized_quant_gb300 import inputs as I
from tests.gpu_util import check_close, dev, gq4_module, host, requires_cuda, tol_fp32

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(scope="module")
def gq4():
    g = gq4_module()
    g.device_error(clear=True)
    return g


def assert_same_params(name, got, ref):
    """Equal values (either zero sign counts as the same value) and NaN where NaN."""
    got, ref = np.asarray(got), np.asarray(ref)
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{name}: NaN positions differ"
    ok = (got == ref) | nan_r
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"{name}: {int((~ok).sum())} differ, first at {tuple(i)}: "
                             f"{got[tuple(i)]!r} vs {ref[tuple(i)]!r}")


def words(t):
    return host(t).view(np.uint32)


QUANT_CASES = [
    # K, N, gs
    (64, 1, 32),
    (256, 33, 32),        # 4 groups per warp task
    (384, 17, 96),        # 12-word groups: 2 per warp task, 8 idle lanes
    (1280, 9, 160),       # 20-word groups
    (1024, 31, 64),
    (4096, 65, 128),
    (512, 31, 256),       # one 32-word group per warp task
    (1152, 3, 288),       # 36 words: the two-pass path
    (2048, 7, 512),
    (4096, 3, 4096),      # one group per column
    (11008, 40, 128),     # the down projection's K
]


@pytest.mark.parametrize("K,N,gs", QUANT_CASES)
def test_quantize(gq4, K, N, gs):
    W = I.float_weights(N, K, 1700, K, N, gs)
    Bq, s, z = gq4.quantize(dev(W), gs)
    torch.cuda.synchronize()
    rBq, rs, rz, bad = oracle.quantize(W, gs)
    assert bad == 0
    assert np.array_equal(words(Bq), rBq)
    assert_same_params("scales", host(s), rs)
    assert_same_params("zeros", host(z), rz)
    assert gq4.device_error() == 0


def test_quantize_gate_up_full(gq4):
    """The 4096 -> 11008 gate/up projection (11008 columns of 4096, gs 128), every
    output compared."""
    K, N, gs = 4096, 11008, 128
    W = I.float_weights(N, K, 1701)
    Bq, s, z = gq4.quantize(dev(W), gs)
    torch.cuda.synchronize()
    rBq, rs, rz, bad = oracle.quantize(W, gs)
    assert bad == 0
    assert np.array_equal(words(Bq), rBq)
    assert_same_params("scales", host(s), rs)
    assert_same_params("zeros", host(z), rz)


# Rows of float_weights(11008, 4096, tag 1701) holding a code whose scaled
# offset t = fl(fl(v - lo) * r) rounds, in binary32, onto or across a half
# integer: rounding the exact product (an FMA) instead of t flips the code.
NEAR_TIE_ROWS = [1746, 6838, 7108, 7768, 7972, 8268, 8314, 10226, 10371, 10735]


def test_quantize_near_ties(gq4):
    """Codes decided by binary32 rounding of t (not of the exact product)."""
    K, gs = 4096, 128
    W = np.ascontiguousarray(I.float_weights(11008, K, 1701)[NEAR_TIE_ROWS])
    Bq, s, z = gq4.quantize(dev(W), gs)
    torch.cuda.synchronize()
    rBq, rs, rz, _ = oracle.quantize(W, gs)
    assert np.array_equal(words(Bq), rBq)
    assert_same_params("scales", host(s), rs)


@pytest.mark.parametrize("gs", [32, 96, 512])
def test_quantize_special_groups(gq4, gs):
    """Constant, all-zero and signed-zero groups, a subnormal range, a NaN, an
    infinity and an overflowing range: the same codes, scales and zeros as the
    oracle, and device error bit 3 exactly when a group is non-finite."""
    K, N = 4 * gs, 8
    W = I.float_weights(N, K, 1702, gs)
    W[0, :gs] = 3.25
    W[1, :] = 0.0
    W[1, gs:2 * gs] = -0.0
    W[1, gs + 1] = 0.0
    W[2, 2 * gs:3 * gs] = np.where(np.arange(gs) % 3 == 0, 1e-40, 2e-40).astype(np.float32)
    W[3, :gs] = np.where(np.arange(gs) % 2 == 0, 3e38, -3e38).astype(np.float32)
    W[4, 5] = np.nan
    W[5, 3 * gs + 7] = np.inf
    W[6, gs] = -np.inf
    W[7, :] = 1e30  # large and constant
    W[7, 2 * gs + 1] = 1e30 * (1 + 2.0 ** -20)
    gq4.device_error(clear=True)
    Bq, s, z = gq4.quantize(dev(W), gs)
    torch.cuda.synchronize()
    rBq, rs, rz, bad = oracle.quantize(W, gs)
    assert bad == 4
    assert np.array_equal(words(Bq), rBq)
    assert_same_params("scales", host(s), rs)
    assert_same_params("zeros", host(z), rz)
    assert gq4.device_error(clear=True) == 1 << 3
    # finite input: the bit stays clear
    W2 = I.float_weights(N, K, 1703, gs)
    gq4.quantize(dev(W2), gs)
    torch.cuda.synchronize()
    assert gq4.device_error() == 0


def test_quantize_round_trip(gq4):
    """Quantize on the GPU, then the library's dequant equals the oracle's binary32
    dequant of the oracle's quantization, bit for bit, and the matvec on the
    quantized weights agrees with the oracle's within the fp32 tolerance."""
    K, N, gs = 2048, 300, 64
    W = I.float_weights(N, K, 1704)
    Bq, s, z = gq4.quantize(dev(W), gs)
    Wd = torch.empty((N, K), dtype=torch.float32, device="cuda")
    gq4.dequant(Bq, s, z, K, gs, W=Wd)
    torch.cuda.synchronize()
    rBq, rs, rz, _ = oracle.quantize(W, gs)
    ref = oracle.dequant_f32(rBq, rs, rz, K, N, gs)
    assert np.array_equal(host(Wd).view(np.uint32), ref.view(np.uint32))
    assert np.all(np.abs(ref.astype(np.float64) - W) <= 0.5 * np.repeat(rs, gs, axis=1) * 1.0001
                  + 4 * 2.0 ** -24 * np.abs(W))
    A = I.activations(1, K, 1704)
    C = host(gq4.matvec(dev(A), Bq, s, z, gs))
    refC, S = oracle.matvec(A, rBq, rs, rz, K, N, gs)
    check_close("matvec of quantized", C, refC, tol_fp32(S))


MLX_CASES = [
    # K, N, gs
    (64, 1, 32),
    (512, 33, 64),
    (384, 17, 96),
    (4096, 65, 128),
    (2048, 9, 512),
]


def _mlx_with_degenerate(K, N, gs, tag):
    m = I.mlx_weights(K, N, gs, tag, K, N, gs)
    s, b = m.scales.copy(), m.biases.copy()
    G = K // gs
    s[0, 0] = 0.0                      # w = bias
    if N > 2:
        s[2, G - 1] = -0.0
        b[2, G - 1] = 0.0
    if N > 3:
        s[3, 0] = 1e-38                # -bias / scale overflows
        b[3, 0] = 3e38
    if N > 4:
        s[4, 0] = np.nan               # propagates
    return m.packed, s, b


@pytest.mark.parametrize("K,N,gs", MLX_CASES)
def test_from_mlx(gq4, K, N, gs):
    packed, s, b = _mlx_with_degenerate(K, N, gs, 1710)
    Bq, sc, z = gq4.from_mlx(dev(packed), dev(s), dev(b), gs)
    torch.cuda.synchronize()
    rBq, rs, rz = oracle.from_mlx(packed, s, b, K, N, gs)
    assert np.array_equal(words(Bq), rBq)
    assert_same_params("scales", host(sc), rs)
    assert_same_params("zeros", host(z), rz)


def test_from_mlx_in_place(gq4):
    """Bq = packed: only the rewritten groups change; the result equals the
    out-of-place conversion."""
    K, N, gs = 1024, 40, 64
    packed, s, b = _mlx_with_degenerate(K, N, gs, 1711)
    words_dev = dev(packed)
    Bq, sc, z = gq4.from_mlx(words_dev, dev(s), dev(b), gs, Bq=words_dev)
    torch.cuda.synchronize()
    assert Bq.data_ptr() == words_dev.data_ptr()
    rBq, rs, rz = oracle.from_mlx(packed, s, b, K, N, gs)
    assert np.array_equal(words(Bq), rBq)
    assert_same_params("scales", host(sc), rs)
    assert_same_params("zeros", host(z), rz)


def _stale_weights(K, N, gs, tag):
    """Device buffers (Bq, scales, zeros) holding other weights, settled before a
    producer overwrites them: a matvec that read them stale fails parity."""
    w = I.quant_weights(K, N, gs, tag, 99)
    bufs = tuple(dev(a) for a in (w.Bq, w.scales, w.zeros))
    torch.cuda.synchronize()
    return bufs


def test_from_mlx_matvec(gq4):
    """gq4_from_mlx immediately followed by gq4_matvec on the same stream (nothing
    in between, no host synchronisation): the matvec streams the converted
    weights, compared with the oracle's matvec of the oracle's conversion."""
    K, N, gs = 4096, 257, 64
    m = I.mlx_weights(K, N, gs, 1712)
    packed, ms, mb = dev(m.packed), dev(m.scales), dev(m.biases)
    Bq, s, z = _stale_weights(K, N, gs, 1712)
    A = dev(I.activations(1, K, 1712))
    C = torch.empty((1, N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        gq4.from_mlx(packed, ms, mb, gs, Bq, s, z)
        gq4.matvec(A, Bq, s, z, gs, C=C)
        torch.cuda.synchronize()
        rBq, rs, rz = oracle.from_mlx(m.packed, m.scales, m.biases, K, N, gs)
        ref, S = oracle.matvec(host(A), rBq, rs, rz, K, N, gs)
        check_close("matvec of converted MLX", host(C), ref, tol_fp32(S))
        # back to stale contents for the next round
        Bq.copy_(_stale_weights(K, N, gs, 1712)[0])
        torch.cuda.synchronize()


def test_quantize_then_matvec_chain(gq4):
    """gq4_quantize immediately followed by gq4_matvec on the same stream (nothing
    in between, no host synchronisation), on the 4096 -> 11008 gate projection:
    the matvec sees the new codes, scales and zeros."""
    K, N, gs = 4096, 11008, 128
    W = dev(I.float_weights(N, K, 1713))
    Bq, s, z = _stale_weights(K, N, gs, 1713)
    A = dev(I.activations(1, K, 1713))
    C = torch.empty((1, N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    gq4.quantize(W, gs, Bq, s, z)
    gq4.matvec(A, Bq, s, z, gs, C=C)
    torch.cuda.synchronize()
    rBq, rs, rz, _ = oracle.quantize(host(W), gs)
    ref, S = oracle.matvec(host(A), rBq, rs, rz, K, N, gs)
    check_close("matvec after quantize", host(C), ref, tol_fp32(S))
    assert gq4.device_error() == 0

"""GPU invariants that hold bit for bit by construction of the kernels.

* quad outputs concatenated == the plain matvec on the same weights;
* lane m of an M-lane call == lane 0 of a smaller call on row m, within one
  kernel: 2..4 lanes (the warp-MMA kernel, gs a multiple of 128: each lane's
  N columns are computed independently) against a two-lane call, 5..15 lanes
  (the CUDA-core kernel, whose per-lane arithmetic does not depend on the
  lane count) against a five-lane call; one-lane calls use the streaming
  kernel and 16..32 lanes the tensor-core kernel, whose orders differ, so
  those are compared within tolerance instead;
* repeated calls give identical bits;
* codes equal to integer zero points give exactly 0 at K = 11008;
* a zero gate gives exactly 0 out of the gated call;
* the gated call equals silu(matvec(gate)) * matvec(up) within tolerance.
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
    return gq4_module()


@pytest.mark.parametrize("M", [1, 3, 8, 16, 32])
def test_quad_equals_matvec(gq4, M):
    K, N, gs = 2560, 1000, 64
    w = I.quant_weights(K, N, gs, 960, M)
    A = dev(I.activations(M, K, 960, M))
    C = host(gq4.matvec(A, *wdev(w), gs))
    for n0, n1, n2 in [(400, 500, 600), (0, 0, 0), (N, N, N), (1, 999, 999), (17, 33, 65)]:
        outs = gq4.quad_matvec(A, *wdev(w), gs, n0, n1, n2)
        cat = np.concatenate([host(o) for o in outs], axis=1)
        assert np.array_equal(cat.view(np.uint32), C.view(np.uint32)), (M, n0, n1, n2)


def _pair(A, m, lanes=2):
    """Rows (m, m+1, ... mod M) of A: a `lanes`-lane call whose lane 0 is row m."""
    return np.ascontiguousarray(A[[(m + i) % A.shape[0] for i in range(lanes)]])


@pytest.mark.parametrize("M", [3, 4, 7, 15])
def test_lane_equals_solo(gq4, M):
    K, N, gs = 4096, 130, 128
    w = I.quant_weights(K, N, gs, 961, M)
    A = I.activations(M, K, 961, M)
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    small = 2 if M <= 4 else 5  # the same kernel as the M-lane call
    for m in range(M):
        Cm = host(gq4.matvec(dev(_pair(A, m, small)), *wdev(w), gs))
        assert np.array_equal(C[m].view(np.uint32), Cm[0].view(np.uint32)), (M, m)
    # and the one-lane streaming kernel agrees with the oracle on every row
    for m in range(min(M, 3)):
        C1 = host(gq4.matvec(dev(A[m:m + 1]), *wdev(w), gs))
        ref, S = oracle.matvec(A[m:m + 1], w.Bq, w.scales, w.zeros, K, N, gs)
        check_close(f"solo row {m}", C1, ref, tol_fp32(S))


def test_norm_lane_equals_solo(gq4):
    M, K, N, gs = 6, 1024, 50, 64
    w = I.quant_weights(K, N, gs, 962)
    A, A_b = I.activations(M, K, 962), I.activations(M, K, 963)
    W = I.norm_gain(K, 962)
    C = host(gq4.norm_matvec(dev(A), *wdev(w), gs, dev(W), 1e-6, A_b=dev(A_b)))
    for m in range(M):
        Cm = host(gq4.norm_matvec(dev(_pair(A, m)), *wdev(w), gs, dev(W), 1e-6,
                                  A_b=dev(_pair(A_b, m))))
        assert np.array_equal(C[m].view(np.uint32), Cm[0].view(np.uint32)), m


def _offset_rows(a, offset_floats=1):
    """A device copy of `a` whose data starts `offset_floats` floats past a 16-byte boundary."""
    import torch
    flat = torch.zeros(a.size + 8, dtype=torch.float32, device="cuda")
    view = flat[offset_floats:offset_floats + a.size].view(*a.shape)
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)).cuda())
    return view


@pytest.mark.parametrize("kind", ["matvec", "quad", "norm", "gated"])
def test_one_lane_general_kernel(gq4, kind):
    """Scale/zero rows that are only 4-byte aligned send a one-lane call to the general
    kernel; both kernels must match the oracle (and each other within tolerance)."""
    M, K, N, gs = 1, 4096, 300, 128
    w = I.quant_weights(K, N, gs, 971)
    wu = I.quant_weights(K, N, gs, 972)
    A = I.activations(M, K, 971)
    A_b = I.activations(M, K, 972)
    W = I.norm_gain(K, 971)
    fast = (dev(w.Bq), dev(w.scales), dev(w.zeros))
    slow = (dev(w.Bq), _offset_rows(w.scales), _offset_rows(w.zeros))
    fast_u = (dev(wu.Bq), dev(wu.scales), dev(wu.zeros))
    slow_u = (dev(wu.Bq), _offset_rows(wu.scales), _offset_rows(wu.zeros))
    if kind == "matvec":
        ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
        outs = [host(gq4.matvec(dev(A), *ws, gs)) for ws in (fast, slow)]
        tol = tol_fp32(S)
    elif kind == "quad":
        ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
        outs = [np.concatenate([host(o) for o in gq4.quad_matvec(dev(A), *ws, gs, 100, 150, 290)],
                               axis=1) for ws in (fast, slow)]
        tol = tol_fp32(S)
    elif kind == "norm":
        ref, S, _, _ = oracle.norm_matvec(A, A_b, W, 1e-6, w.Bq, w.scales, w.zeros, K, N, gs)
        outs = [host(gq4.norm_matvec(dev(A), *ws, gs, dev(W), 1e-6, A_b=dev(A_b)))
                for ws in (fast, slow)]
        tol = tol_fp32(S)
    else:
        r = oracle.gated_matvec(A, w.Bq, w.scales, w.zeros, wu.Bq, wu.scales, wu.zeros, K, N, gs)
        ref = r["out"]
        outs = [host(gq4.gated_matvec(dev(A), *ws, *wsu, gs))
                for ws, wsu in ((fast, fast_u), (slow, slow_u))]
        from tests.gpu_util import tol_gated
        tol = tol_gated(r["g"], r["u"], r["Sg"], r["Su"], ref)
    for name, o in zip(("streaming", "general"), outs):
        check_close(f"{kind} {name}", o, ref, tol)
    assert gq4.device_error() == 0


@pytest.mark.parametrize("N", [1, 3, 7, 150, 151, 300, 301, 4097])
def test_streaming_column_splits(gq4, N):
    """Column counts below, at and above the grid size, odd counts with 86 groups per
    column (scale rows split in units of two columns, a tail read directly)."""
    K, gs = 11008, 128
    w = I.quant_weights(K, N, gs, 973, N)
    A = I.activations(1, K, 973, N)
    ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    check_close(f"stream N={N}", C, ref, tol_fp32(S))
    assert gq4.device_error() == 0


@pytest.mark.parametrize("M", [1, 4, 16, 32])
def test_deterministic(gq4, M):
    K, N, gs = 4096, 1000, 128
    w = I.quant_weights(K, N, gs, 963)
    A = dev(I.activations(M, K, 963))
    first = host(gq4.matvec(A, *wdev(w), gs))
    for _ in range(5):
        again = host(gq4.matvec(A, *wdev(w), gs))
        assert np.array_equal(first.view(np.uint32), again.view(np.uint32))


@pytest.mark.parametrize("M", [1, 4, 16, 32])
def test_zero_point_codes_give_exact_zero(gq4, M):
    K, N, gs = 11008, 70, 128
    G = K // gs
    c = I.rng(964, M).integers(0, 16, size=(N, G)).astype(np.uint32)
    # every code of a group equals the group's integer zero point
    words = np.repeat(c * np.uint32(0x11111111), gs // 8, axis=1).astype(np.uint32)
    zeros = c.astype(np.float32)
    scales = I.uniform_f32((N, G), 0.005, 0.02, 964)
    A = I.activations(M, K, 964, M)
    C = host(gq4.matvec(dev(A), dev(words), dev(scales), dev(zeros), gs))
    assert np.all(C == 0.0), float(np.abs(C).max())
    # the oracle agrees exactly
    C_ref, S = oracle.matvec(A, words, scales, zeros, K, N, gs)
    assert np.all(C_ref == 0.0) and np.all(S == 0.0)


def test_zero_gate_gives_zero(gq4):
    M, K, N, gs = 2, 4096, 300, 128
    G = K // gs
    gate_words = np.full((N, K // 8), 0x77777777, np.uint32)
    gate_zeros = np.full((N, G), 7.0, np.float32)
    gate_scales = I.uniform_f32((N, G), 0.002, 0.01, 965)
    wu = I.quant_weights(K, N, gs, 966)
    A = dev(I.activations(M, K, 965))
    out = host(gq4.gated_matvec(A, dev(gate_words), dev(gate_scales), dev(gate_zeros),
                                *wdev(wu), gs))
    assert np.all(out == 0.0)


def test_gated_is_silu_of_matvecs(gq4):
    M, K, N, gs = 3, 4096, 500, 128
    wg = I.quant_weights(K, N, gs, 967, scale_range=I.SCALE_RANGE_GATED)
    wu = I.quant_weights(K, N, gs, 968, scale_range=I.SCALE_RANGE_GATED)
    A = dev(I.activations(M, K, 967))
    g = host(gq4.matvec(A, *wdev(wg), gs)).astype(np.float64)
    u = host(gq4.matvec(A, *wdev(wu), gs)).astype(np.float64)
    out = host(gq4.gated_matvec(A, *wdev(wg), *wdev(wu), gs)).astype(np.float64)
    expect = g / (1.0 + np.exp(-g)) * u
    # same dot products bit for bit; only expf / division / product rounding differ
    check_close("gated vs composed", out, expect, 4e-7 * np.abs(expect) + 1e-9)


def test_nonfinite_activation_propagates(gq4):
    """An Inf or NaN activation poisons exactly the outputs it feeds (no silent masking)."""
    M, K, N, gs = 2, 256, 40, 32
    w = I.quant_weights(K, N, gs, 969)
    A = I.activations(M, K, 969)
    A[1, 5] = np.nan
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    assert np.all(np.isfinite(C[0])) and np.all(np.isnan(C[1]))


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_one_lane_nonfinite_activation(gq4, bad):
    """M = 1 (the integer one-lane path): a NaN or infinite activation makes
    every output NaN (each column's dot product uses it), nothing is masked."""
    K, N, gs = 4096, 300, 128
    w = I.quant_weights(K, N, gs, 971)
    A = I.activations(1, K, 971)
    A[0, 777] = bad
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    assert np.all(np.isnan(C))


@pytest.mark.parametrize("outlier,scale", [(100.0, 1.0), (1000.0, 1.0), (1.0, 1e-30), (1.0, 1e20)])
def test_one_lane_activation_dynamic_range(gq4, outlier, scale):
    """M = 1 holds activations as 24-bit fixed point per 64-code group (a
    power-of-two scale per group): one outlier of 100x or 1000x the typical
    magnitude in every group, and vectors scaled to 1e-30 or 1e20, stay
    within the fp32 tolerance against the oracle."""
    K, N, gs = 4096, 512, 128
    w = I.quant_weights(K, N, gs, 972, int(outlier))
    A = I.activations(1, K, 972, int(outlier)) * np.float32(scale)
    r = np.random.default_rng(973)
    pos = np.arange(0, K, 64) + r.integers(0, 64, size=K // 64)
    A[0, pos] = np.float32(outlier * scale) * np.sign(r.standard_normal(pos.size)).astype(np.float32)
    A = A.astype(np.float32)
    C = host(gq4.matvec(dev(A), *wdev(w), gs))
    ref, S = oracle.matvec(A, w.Bq, w.scales, w.zeros, K, N, gs)
    check_close(f"outlier {outlier} scale {scale}", C, ref, tol_fp32(S))


def test_stream_argument(gq4):
    """Calls run on the stream they are given and respect its ordering."""
    M, K, N, gs = 1, 1024, 1024, 32
    w = I.quant_weights(K, N, gs, 970)
    A = I.activations(M, K, 970)
    ref = host(gq4.matvec(dev(A), *wdev(w), gs))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Ad = dev(A)
        out = gq4.matvec(Ad, *wdev(w), gs, stream=s)
    s.synchronize()
    assert np.array_equal(host(out).view(np.uint32), ref.view(np.uint32))

"""Pins for the oracle: facts fixed by the pages and by mathematics.

Each ``pin_*`` takes an oracle instance and raises ``AssertionError`` if the
oracle disagrees with something that does not depend on the oracle itself:

* an independent byte-view unpack of the word layout (little-endian bytes,
  element k of a column is byte k/2 of the column, low nibble when k is even);
* fixed words whose codes are known by construction;
* one-hot activations, which must return one dequantized weight exactly;
* exact rational brute force (Python ``fractions``) on dyadic inputs;
* all codes equal to integer zero points, which must give exactly 0;
* split-routing invariants of the quad matvec;
* closed forms of the RMSNorm prologue and SiLU-gated epilogue.

The pins are also run against deliberately broken copies of the oracle
(``tests/test_oracle_mutants.py``) to show that each planted mistake fails at
least one of them.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


# ---------------------------------------------------------------------------
# Independent helpers (no oracle code): byte-view unpack and dyadic inputs.
# ---------------------------------------------------------------------------

def byte_view_codes(Bq: np.ndarray, K: int, N: int) -> np.ndarray:
    """Codes [N, K] read through a little-endian byte view of the words."""
    b = np.ascontiguousarray(Bq.astype("<u4")).view(np.uint8).reshape(N, K // 2)
    out = np.empty((N, K), np.uint8)
    out[:, 0::2] = b & 0x0F
    out[:, 1::2] = b >> 4
    return out


def _rng(seed):
    return np.random.default_rng(seed)


def _dyadic_problem(seed, M, K, N, gs):
    """Inputs whose every product and partial sum is exact in double."""
    r = _rng(seed)
    G = K // gs
    Bq = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    scales = (2.0 ** r.integers(-3, 4, size=(N, G))).astype(np.float32)
    zeros = (r.integers(0, 31, size=(N, G)) * 0.5).astype(np.float32)  # 0, 0.5, ..., 15
    A = r.integers(-8, 9, size=(M, K)).astype(np.float32)
    return A, Bq, scales, zeros


def _fraction_matvec(A, codes, scales, zeros, gs):
    """C[m][n] = sum_k A[m,k] (q - z) s over exact rationals."""
    M, K = A.shape
    N = codes.shape[0]
    C = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        w = [(Fraction(int(codes[n, k])) - Fraction(float(zeros[n, k // gs])))
             * Fraction(float(scales[n, k // gs])) for k in range(K)]
        for m in range(M):
            C[m][n] = sum((Fraction(float(A[m, k])) * w[k] for k in range(K)), Fraction(0))
    return C


# ---------------------------------------------------------------------------
# Layout pins
# ---------------------------------------------------------------------------

def pin_fixed_words(orc):
    """0x76543210 holds codes 0..7 and 0xFEDCBA98 codes 8..15, lowest nibble first."""
    words = np.array([[0x76543210, 0xFEDCBA98, 0x00000000, 0xFFFFFFFF]], np.uint32)
    q = orc.unpack(words, 32, 1)[0]
    assert list(q[0:8]) == list(range(8)), q[0:8]
    assert list(q[8:16]) == list(range(8, 16)), q[8:16]
    assert list(q[16:24]) == [0] * 8
    assert list(q[24:32]) == [15] * 8
    # element-wise accessor agrees
    for k in range(32):
        assert orc.nibble(words, 32, 0, k) == int(q[k])


def pin_byte_view(orc):
    """The oracle's unpack agrees with an independent little-endian byte view."""
    for seed, (K, N) in enumerate([(8, 1), (32, 3), (64, 5), (1024, 7)]):
        Bq = _rng(seed).integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
        assert np.array_equal(orc.unpack(Bq, K, N), byte_view_codes(Bq, K, N))


def pin_pack_round_trip(orc):
    """pack then unpack is the identity on codes; unpack then pack on words."""
    for seed, (K, N) in enumerate([(8, 1), (40, 3), (256, 9)]):
        q = _rng(100 + seed).integers(0, 16, size=(N, K), dtype=np.uint8)
        Bq = orc.pack(q)
        assert np.array_equal(orc.unpack(Bq, K, N), q)
        assert np.array_equal(orc.pack(orc.unpack(Bq, K, N)), Bq)
        assert np.array_equal(byte_view_codes(Bq, K, N), q)


# ---------------------------------------------------------------------------
# Dequant and dot-product pins
# ---------------------------------------------------------------------------

def pin_one_hot(orc):
    """A = e_k returns w(n,k) = (q - z) s exactly, across group boundaries."""
    K, N, gs = 256, 6, 64
    r = _rng(7)
    Bq = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    scales = r.uniform(0.005, 0.02, size=(N, K // gs)).astype(np.float32)
    zeros = r.uniform(6, 9, size=(N, K // gs)).astype(np.float32)
    codes = byte_view_codes(Bq, K, N).astype(np.float64)
    s_full = np.repeat(scales.astype(np.float64), gs, axis=1)
    z_full = np.repeat(zeros.astype(np.float64), gs, axis=1)
    W_expect = (codes - z_full) * s_full          # exact in double
    for k in [0, 1, 7, 8, gs - 1, gs, gs + 1, 2 * gs - 1, 2 * gs, K - 1]:
        A = np.zeros((1, K), np.float32)
        A[0, k] = 1.0
        C, S = orc.matvec(A, Bq, scales, zeros, K, N, gs)
        assert np.array_equal(C[0], W_expect[:, k]), (k, C[0], W_expect[:, k])
        assert np.array_equal(S[0], np.abs(W_expect[:, k]))
    assert np.array_equal(orc.dequant_f64(Bq, scales, zeros, K, N, gs), W_expect)


def pin_dequant_f32(orc):
    """The binary32 dequant equals numpy's binary32 (q - z) then * s, bit for bit."""
    K, N, gs = 512, 9, 32
    r = _rng(8)
    Bq = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    scales = r.uniform(0.005, 0.02, size=(N, K // gs)).astype(np.float32)
    zeros = r.uniform(6, 9, size=(N, K // gs)).astype(np.float32)
    codes = byte_view_codes(Bq, K, N).astype(np.float32)
    t = (codes - np.repeat(zeros, gs, axis=1)).astype(np.float32)
    w = (t * np.repeat(scales, gs, axis=1)).astype(np.float32)
    got = orc.dequant_f32(Bq, scales, zeros, K, N, gs)
    assert np.array_equal(got.view(np.uint32), w.view(np.uint32))


def pin_brute_force_exact(orc):
    """Exact rational brute force on dyadic inputs (every term exact in double)."""
    cases = [(1, 32, 1, 32), (2, 32, 3, 8), (1, 64, 5, 32), (3, 128, 9, 64),
             (2, 128, 4, 16), (1, 96, 2, 32)]
    for seed, (M, K, N, gs) in enumerate(cases):
        A, Bq, scales, zeros = _dyadic_problem(200 + seed, M, K, N, gs)
        C, _ = orc.matvec(A, Bq, scales, zeros, K, N, gs)
        exact = _fraction_matvec(A, byte_view_codes(Bq, K, N), scales, zeros, gs)
        for m in range(M):
            for n in range(N):
                assert Fraction(float(C[m, n])) == exact[m][n], (M, K, N, gs, m, n)


def pin_abs_sum(orc):
    """S = sum |a w|: with all activations positive and all weights positive, S = C."""
    K, N, gs = 64, 4, 32
    r = _rng(9)
    q = np.full((N, K), 12, np.uint8)
    Bq = orc.pack(q)
    scales = r.uniform(0.5, 1.0, size=(N, K // gs)).astype(np.float32)
    zeros = np.full((N, K // gs), 3.0, np.float32)  # q - z = 9 > 0
    A = r.uniform(0.1, 1.0, size=(1, K)).astype(np.float32)
    C, S = orc.matvec(A, Bq, scales, zeros, K, N, gs)
    assert np.allclose(C, S, rtol=1e-15, atol=0)
    C2, S2 = orc.matvec(-A, Bq, scales, zeros, K, N, gs)
    assert np.array_equal(C2, -C) and np.array_equal(S2, S)


def pin_zero_point_exact(orc):
    """Every code equal to its group's integer zero point gives exactly 0 (K = 11008)."""
    K, N, gs = 11008, 3, 128
    r = _rng(10)
    G = K // gs
    c = r.integers(0, 16, size=(N, G))
    codes = np.repeat(c, gs, axis=1).astype(np.uint8)
    Bq = orc.pack(codes)
    zeros = c.astype(np.float32)
    scales = r.uniform(0.005, 0.02, size=(N, G)).astype(np.float32)
    A = r.standard_normal((2, K)).astype(np.float32)
    C, S = orc.matvec(A, Bq, scales, zeros, K, N, gs)
    assert np.all(C == 0.0) and np.all(S == 0.0)


def pin_lanes_independent(orc):
    """Lane m of an M-lane call equals the one-lane call on row m, bit for bit."""
    K, N, gs = 256, 5, 64
    r = _rng(11)
    Bq = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    scales = r.uniform(0.005, 0.02, size=(N, K // gs)).astype(np.float32)
    zeros = r.uniform(6, 9, size=(N, K // gs)).astype(np.float32)
    A = r.standard_normal((4, K)).astype(np.float32)
    C, _ = orc.matvec(A, Bq, scales, zeros, K, N, gs)
    for m in range(4):
        Cm, _ = orc.matvec(A[m:m + 1], Bq, scales, zeros, K, N, gs)
        assert np.array_equal(C[m], Cm[0])
    # and the double-activation column sampler agrees with the f32 path
    Cc, _ = orc.dot_cols(A.astype(np.float64), Bq, scales, zeros, K, gs, [4, 0, 2])
    assert np.array_equal(Cc, C[:, [4, 0, 2]])


# ---------------------------------------------------------------------------
# Quad routing
# ---------------------------------------------------------------------------

def pin_quad_routing(orc):
    """concat(out0..out3) equals the unsplit matvec for many split points."""
    K, N, gs = 64, 11, 32
    r = _rng(12)
    Bq = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    scales = r.uniform(0.005, 0.02, size=(N, K // gs)).astype(np.float32)
    zeros = r.uniform(6, 9, size=(N, K // gs)).astype(np.float32)
    A = r.standard_normal((2, K)).astype(np.float32)
    C, S = orc.matvec(A, Bq, scales, zeros, K, N, gs)
    splits = [(4, 6, 8), (0, 0, 0), (0, 0, N), (N, N, N), (1, 2, 3), (0, 5, 5),
              (3, 3, 10), (10, 10, 11), (2, 9, 9)]
    for n0, n1, n2 in splits:
        outs, sabs = orc.quad_matvec(A, Bq, scales, zeros, K, N, gs, n0, n1, n2)
        assert [o.shape[1] for o in outs] == [n0, n1 - n0, n2 - n1, N - n2]
        assert np.array_equal(np.concatenate(outs, axis=1), C), (n0, n1, n2)
        assert np.array_equal(np.concatenate(sabs, axis=1), S)


# ---------------------------------------------------------------------------
# RMSNorm prologue
# ---------------------------------------------------------------------------

def pin_norm_constant(orc):
    """A_a = c, A_b = 0, W = 1: a_k = c / sqrt(c^2 + eps) (closed form, high precision)."""
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    K = 256
    for c, eps in [(0.5, 1e-6), (3.0, 1e-6), (-2.0, 0.25), (1e-3, 1e-6)]:
        A_a = np.full((1, K), c, np.float32)
        A_b = np.zeros((1, K), np.float32)
        W = np.ones(K, np.float32)
        x, a, inv = orc.norm(A_a, A_b, W, eps, K)
        cf = Decimal(float(np.float32(c)))
        ef = Decimal(float(np.float32(eps)))
        expect = float(cf / (cf * cf + ef).sqrt())
        assert np.all(x == np.float32(c))
        # the oracle's K-term double sum of x^2 carries at most ~K ulps of error
        assert np.allclose(a, expect, rtol=(K + 8) * 2.0 ** -53, atol=0), (c, eps, a[0, 0], expect)


def pin_norm_gain_closed_form(orc):
    """A_a = c, A_b = 0 and a gain of distinct powers of two (then one-hot):
    a_k = c * W_k / sqrt(c^2 + eps) element by element (closed form, 50 digits).

    Every W_k differs from its neighbours, so a dropped gain, a gain read at
    the wrong index or a gain applied once for the whole vector each fail."""
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    K = 96
    gains = [np.float32(2.0 ** ((k * 5) % 11 - 5)) for k in range(K)]
    one_hot = [np.float32(0.0)] * K
    one_hot[37] = np.float32(8.0)
    for c, eps, W in [(0.75, 1e-6, gains), (-3.0, 0.5, gains), (2.0, 1e-6, one_hot)]:
        A_a = np.full((1, K), c, np.float32)
        A_b = np.zeros((1, K), np.float32)
        Wv = np.array(W, np.float32)
        x, a, _ = orc.norm(A_a, A_b, Wv, eps, K)
        cf = Decimal(float(np.float32(c)))
        base = cf / (cf * cf + Decimal(float(np.float32(eps)))).sqrt()
        expect = np.array([float(base * Decimal(float(w))) for w in W])
        assert np.all(x == np.float32(c))
        assert np.all(np.abs(a[0] - expect) <= (K + 8) * 2.0 ** -53 * np.abs(expect)), (c, eps)


def pin_norm_scale_invariance(orc):
    """With eps = 0, doubling x leaves the normalised vector unchanged exactly."""
    K = 512
    r = _rng(13)
    A_a = r.standard_normal((2, K)).astype(np.float32)
    W = r.uniform(0.5, 1.5, size=K).astype(np.float32)
    _, a1, inv1 = orc.norm(A_a, None, W, 0.0, K)
    _, a2, inv2 = orc.norm(2 * A_a, None, W, 0.0, K)
    assert np.array_equal(a1, a2)
    assert np.array_equal(inv1, 2 * inv2)
    # unit gain, eps 0: the normalised vector has mean square 1
    _, a3, _ = orc.norm(A_a, None, np.ones(K, np.float32), 0.0, K)
    assert np.allclose(np.mean(a3 ** 2, axis=1), 1.0, rtol=1e-13)


def pin_norm_residual(orc):
    """residual_out is the binary32 sum A_a + A_b, bit for bit; C uses the normalised a."""
    K, N, gs = 256, 4, 64
    r = _rng(14)
    A_a = r.standard_normal((3, K)).astype(np.float32)
    A_b = r.standard_normal((3, K)).astype(np.float32)
    W = r.uniform(0.5, 1.5, size=K).astype(np.float32)
    Bq = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    scales = r.uniform(0.005, 0.02, size=(N, K // gs)).astype(np.float32)
    zeros = r.uniform(6, 9, size=(N, K // gs)).astype(np.float32)
    C, S, res, nout = orc.norm_matvec(A_a, A_b, W, 1e-6, Bq, scales, zeros, K, N, gs)
    assert np.array_equal(res.view(np.uint32), (A_a + A_b).astype(np.float32).view(np.uint32))
    Cd, Sd = orc.dot_cols(nout, Bq, scales, zeros, K, gs, list(range(N)))
    assert np.array_equal(C, Cd) and np.array_equal(S, Sd)
    # the normalised activation: x * inv * W with inv from the mean of x^2 over K
    x64 = res.astype(np.float64)
    inv = 1.0 / np.sqrt(np.mean(x64 * x64, axis=1) + float(np.float32(1e-6)))
    assert np.allclose(nout, x64 * inv[:, None] * W.astype(np.float64), rtol=1e-13, atol=0)


# ---------------------------------------------------------------------------
# SiLU-gated gate/up
# ---------------------------------------------------------------------------

def _silu(t):
    return t / (1.0 + math.exp(-t)) if t > -700 else 0.0


def pin_gated_closed_forms(orc):
    """All-ones up matrix gives u = sum(a); zero gate gives out = 0; silu(g) * u otherwise."""
    K, N, gs = 128, 6, 32
    r = _rng(15)
    G = K // gs
    A = r.standard_normal((2, K)).astype(np.float32)
    # up: every code 5, zero 4, scale 1  -> w = 1 exactly
    Bu = orc.pack(np.full((N, K), 5, np.uint8))
    su = np.ones((N, G), np.float32)
    zu = np.full((N, G), 4.0, np.float32)
    # gate: random
    Bg = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    sg = r.uniform(0.002, 0.01, size=(N, G)).astype(np.float32)
    zg = r.uniform(6, 9, size=(N, G)).astype(np.float32)
    res = orc.gated_matvec(A, Bg, sg, zg, Bu, su, zu, K, N, gs)
    asum = A.astype(np.float64).sum(axis=1)
    assert np.allclose(res["u"], asum[:, None], rtol=1e-14, atol=1e-14)
    Cg, _ = orc.matvec(A, Bg, sg, zg, K, N, gs)
    assert np.array_equal(res["g"], Cg)
    expect = np.vectorize(_silu)(Cg) * res["u"]
    assert np.allclose(res["out"], expect, rtol=1e-15, atol=0)
    # zero gate: codes equal to integer zero points
    Bz = orc.pack(np.full((N, K), 7, np.uint8))
    zz = np.full((N, G), 7.0, np.float32)
    res0 = orc.gated_matvec(A, Bz, sg, zz, Bg, sg, zg, K, N, gs)
    assert np.all(res0["out"] == 0.0) and np.all(res0["g"] == 0.0)


def pin_silu_values(orc):
    """silu at known points through a one-weight gate and unit up: out = silu(t)."""
    K, N, gs = 8, 1, 8
    Bq_one = orc.pack(np.full((N, K), 1, np.uint8))        # q = 1
    z0 = np.zeros((1, 1), np.float32)
    s1 = np.ones((1, 1), np.float32)
    for t, expect in [(0.0, 0.0), (1.0, 1.0 / (1.0 + math.exp(-1.0))),
                      (-1.0, -1.0 / (1.0 + math.e)), (20.0, 20.0 / (1.0 + math.exp(-20.0))),
                      (-800.0, -0.0)]:
        A = np.zeros((1, K), np.float32)
        A[0, 0] = t
        # gate weights: only element 0 is 1 (others q=0 with zero 0 -> 0); up: all ones
        codes = np.zeros((N, K), np.uint8)
        codes[0, 0] = 1
        Bg = orc.pack(codes)
        res = orc.gated_matvec(A, Bg, s1, z0, Bq_one, s1, z0, K, N, gs)
        assert res["g"][0, 0] == t and res["u"][0, 0] == t
        assert res["out"][0, 0] == expect * t or math.isclose(
            res["out"][0, 0], expect * t, rel_tol=1e-15), (t, res["out"][0, 0])


def pin_gated_norm(orc):
    """The gated call with a norm prologue equals gated on the oracle's normalised a."""
    K, N, gs = 256, 5, 64
    r = _rng(16)
    G = K // gs
    A = r.standard_normal((2, K)).astype(np.float32)
    A_b = r.standard_normal((2, K)).astype(np.float32)
    W = r.uniform(0.5, 1.5, size=K).astype(np.float32)
    Bg = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    Bu = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    sg = r.uniform(0.002, 0.01, size=(N, G)).astype(np.float32)
    su = r.uniform(0.002, 0.01, size=(N, G)).astype(np.float32)
    zg = r.uniform(6, 9, size=(N, G)).astype(np.float32)
    zu = r.uniform(6, 9, size=(N, G)).astype(np.float32)
    res = orc.gated_matvec(A, Bg, sg, zg, Bu, su, zu, K, N, gs, A_b=A_b, W_norm=W, eps=1e-6)
    x, a, _ = orc.norm(A, A_b, W, 1e-6, K)
    assert np.array_equal(res["residual_out"], x)
    assert np.array_equal(res["norm_out"], a)
    g, _ = orc.dot_cols(a, Bg, sg, zg, K, gs, list(range(N)))
    u, _ = orc.dot_cols(a, Bu, su, zu, K, gs, list(range(N)))
    assert np.array_equal(res["g"], g) and np.array_equal(res["u"], u)


# ---------------------------------------------------------------------------
# Gated input (GatedMatVecInt4: x * sigmoid(g); SwiGLUGatedMatVecInt4: silu(g) * x)
# ---------------------------------------------------------------------------

def _gated_input_problem(seed, M=2, K=256, N=9, gs=64):
    r = _rng(seed)
    G = K // gs
    X = r.standard_normal((M, K)).astype(np.float32)
    Bq = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    s = r.uniform(0.005, 0.02, size=(N, G)).astype(np.float32)
    z = r.uniform(6, 9, size=(N, G)).astype(np.float32)
    return X, Bq, s, z, K, N, gs


def pin_gated_input_saturation(orc):
    """sigmoid(0) = 1/2 halves the matvec exactly; a gate of 64 saturates sigmoid to 1
    (the plain matvec) and silu to 64 (64 times it), exactly in double; silu(0) gives 0."""
    X, Bq, s, z, K, N, gs = _gated_input_problem(17)
    C0, S0 = orc.matvec(X, Bq, s, z, K, N, gs)
    zero = np.zeros_like(X)
    big = np.full_like(X, 64.0)
    C, S, a = orc.gated_input_matvec("sigmoid", X, zero, Bq, s, z, K, N, gs)
    assert np.array_equal(C, 0.5 * C0) and np.array_equal(S, 0.5 * S0)
    assert np.array_equal(a, 0.5 * X.astype(np.float64))
    C, S, _ = orc.gated_input_matvec("sigmoid", X, big, Bq, s, z, K, N, gs)
    assert np.array_equal(C, C0) and np.array_equal(S, S0)
    C, S, _ = orc.gated_input_matvec("swiglu", X, big, Bq, s, z, K, N, gs)
    assert np.array_equal(C, 64.0 * C0) and np.array_equal(S, 64.0 * S0)
    C, S, _ = orc.gated_input_matvec("swiglu", X, zero, Bq, s, z, K, N, gs)
    assert np.all(C == 0.0) and np.all(S == 0.0)


def pin_gated_input_values(orc):
    """Through a one-hot weight (w = 1 at k = 0), the input element is returned:
    sigmoid and silu at known points, and the roles of x and g are not swapped."""
    K, N, gs = 8, 1, 8
    codes = np.zeros((N, K), np.uint8)
    codes[0, 0] = 1
    Bq = orc.pack(codes)
    s1 = np.ones((1, 1), np.float32)
    z0 = np.zeros((1, 1), np.float32)
    for x, g in [(1.0, 0.0), (2.0, 1.0), (-3.0, -1.0), (0.5, 20.0), (4.0, -2.5)]:
        X = np.zeros((1, K), np.float32)
        Gt = np.zeros((1, K), np.float32)
        X[0, 0], Gt[0, 0] = x, g
        sig = 1.0 / (1.0 + math.exp(-g))
        C, _, _ = orc.gated_input_matvec("sigmoid", X, Gt, Bq, s1, z0, K, N, gs)
        assert math.isclose(C[0, 0], x * sig, rel_tol=1e-15), (x, g, C[0, 0])
        C, _, _ = orc.gated_input_matvec("swiglu", X, Gt, Bq, s1, z0, K, N, gs)
        assert math.isclose(C[0, 0], g * sig * x, rel_tol=1e-15), (x, g, C[0, 0])


# ---------------------------------------------------------------------------
# Quantizer and MLX conversion
# ---------------------------------------------------------------------------

_U = 2.0 ** -24  # unit roundoff of binary32


def _group_view(x, gs):
    N, K = x.shape
    return x.reshape(N, K // gs, gs)


def pin_quantize_grid(orc):
    """Values on a 16-level grid lo + j*s (power-of-two s, lo a multiple of s,
    both ends in every group) come back exactly: codes j, scale s, zero -lo/s,
    and the dequantized values.  A group size of 96 (12 words) included."""
    r = _rng(30)
    N, K, gs = 5, 384, 96
    G = K // gs
    codes = r.integers(0, 16, size=(N, K)).astype(np.uint8)
    for g in range(G):
        codes[:, g * gs + 3] = 0
        codes[:, g * gs + 50] = 15
    s = 2.0 ** r.integers(-8, 3, size=(N, G))
    j = r.integers(-20, 6, size=(N, G))
    W = (j * s)[:, :, None] + _group_view(codes, gs) * s[:, :, None]
    W = W.reshape(N, K).astype(np.float32)
    Bq, sc, z, bad = orc.quantize(W, gs)
    assert bad == 0
    assert np.array_equal(byte_view_codes(Bq, K, N), codes)
    assert np.array_equal(sc, s.astype(np.float32))
    assert np.array_equal(z, (-j).astype(np.float32))
    assert np.array_equal(orc.dequant_f64(Bq, sc, z, K, N, gs), W.astype(np.float64))


def pin_quantize_nearest(orc):
    """Random groups: every code is the nearest of its group's 16 levels
    (q - z) * s (brute force over the 16, in double), the error is at most
    half a step, codes 0 and 15 both occur, and the levels of codes 0 and 15
    are the group's min and max to within rounding."""
    r = _rng(31)
    N, K, gs = 7, 512, 128
    W = (r.normal(0.0, 0.02, size=(N, K)) + r.normal(0.0, 0.01, size=(N, 1))).astype(np.float32)
    Bq, s, z, bad = orc.quantize(W, gs)
    assert bad == 0
    codes = byte_view_codes(Bq, K, N).astype(np.int64)
    sd = np.repeat(s.astype(np.float64), gs, axis=1)
    zd = np.repeat(z.astype(np.float64), gs, axis=1)
    levels = (np.arange(16)[None, None, :] - zd[:, :, None]) * sd[:, :, None]
    err = np.abs(W.astype(np.float64)[:, :, None] - levels)
    mine = np.take_along_axis(err, codes[:, :, None], axis=2)[:, :, 0]
    assert np.all(mine <= err.min(axis=2) + 1e-5 * sd)
    assert np.all(mine <= 0.5 * sd * (1.0 + 1e-5))
    cg = _group_view(codes, gs)
    assert np.all(cg.min(axis=2) == 0) and np.all(cg.max(axis=2) == 15)
    Wg = _group_view(W.astype(np.float64), gs)
    lo, hi = Wg.min(axis=2), Wg.max(axis=2)
    s64, z64 = s.astype(np.float64), z.astype(np.float64)
    tol = 4 * _U * (np.abs(lo) + np.abs(hi))
    assert np.all(np.abs((0.0 - z64) * s64 - lo) <= tol)
    assert np.all(np.abs((15.0 - z64) * s64 - hi) <= tol)


def pin_quantize_special_groups(orc):
    """A constant group dequantizes to exactly its value (scale 1), an all-zero
    group to 0; a subnormal range falls back to scale 1 with the minimum
    reproduced; a group holding NaN or inf, or whose range overflows, is
    counted and gets codes 0 and a NaN scale and zero, without touching the
    other group of its column."""
    K, gs, N = 64, 32, 6
    r = _rng(33)
    W = r.normal(0.0, 1.0, size=(N, K)).astype(np.float32)
    W[0] = 3.25
    W[1] = 0.0
    W[2, 5] = np.nan
    W[3, 40] = np.inf
    W[4, :32] = np.where(np.arange(32) % 2 == 0, 3e38, -3e38).astype(np.float32)
    W[5, :32] = np.where(np.arange(32) % 3 == 0, 1e-40, 2e-40).astype(np.float32)
    Bq, s, z, bad = orc.quantize(W, gs)
    assert bad == 3
    codes = byte_view_codes(Bq, K, N)
    D = orc.dequant_f64(Bq, s, z, K, N, gs)
    assert np.all(D[0] == 3.25) and np.all(s[0] == 1.0)
    assert np.all(D[1] == 0.0)
    for n, g in ((2, 0), (3, 1), (4, 0)):
        assert math.isnan(s[n, g]) and math.isnan(z[n, g])
        assert np.all(codes[n, g * gs:(g + 1) * gs] == 0)
        other = 1 - g
        seg = slice(other * gs, (other + 1) * gs)
        assert np.isfinite(s[n, other])
        assert np.all(np.abs(D[n, seg] - W[n, seg]) <= 0.5 * s[n, other] * (1 + 1e-5)
                      + 4 * _U * np.abs(W[n, seg]).max())
    assert s[5, 0] == 1.0 and D[5, 0] == np.float64(np.float32(1e-40))


def pin_mlx_worked_example(orc):
    """MLX words 0x76543210 and 0xFEDCBA98 (codes 0..7 and 8..15) with scale 1/2
    and bias -4 give w = q/2 - 4 = -4, -3.5, ..., 3.5, through the page's
    formula and through the conversion (zero 8) and this format's dequant."""
    K, N, gs = 32, 1, 32
    packed = np.array([[0x76543210, 0xFEDCBA98, 0x76543210, 0xFEDCBA98]], np.uint32)
    ms = np.array([[0.5]], np.float32)
    mb = np.array([[-4.0]], np.float32)
    expect = np.array([q / 2.0 - 4.0 for q in list(range(16)) * 2])
    assert np.array_equal(orc.mlx_dequant_f64(packed, ms, mb, K, N, gs)[0], expect)
    Bq, s, z = orc.from_mlx(packed, ms, mb, K, N, gs)
    assert np.array_equal(Bq, packed) and s[0, 0] == 0.5 and z[0, 0] == 8.0
    assert np.array_equal(orc.dequant_f64(Bq, s, z, K, N, gs)[0], expect)


def _mlx_problem(seed, N=6, K=256, gs=64):
    r = _rng(seed)
    G = K // gs
    packed = r.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    ms = (r.uniform(1e-3, 1e-2, size=(N, G)) * r.choice([-1.0, 1.0], size=(N, G)))
    mb = -np.abs(ms) * r.uniform(0.0, 15.0, size=(N, G)) + r.normal(0.0, 1e-3, size=(N, G))
    return packed, ms.astype(np.float32), mb.astype(np.float32), K, N, gs


def pin_mlx_conversion(orc):
    """Random MLX matrices: codes and scales pass through, and this format's
    dequant of the conversion equals the page's scale * q + bias to within the
    one rounding of the zero, |error| <= 2^-24 |bias| (in double both sides
    are otherwise exact)."""
    packed, ms, mb, K, N, gs = _mlx_problem(34)
    Bq, s, z = orc.from_mlx(packed, ms, mb, K, N, gs)
    assert np.array_equal(Bq, packed) and np.array_equal(s, ms)
    D = orc.dequant_f64(Bq, s, z, K, N, gs)
    R = orc.mlx_dequant_f64(packed, ms, mb, K, N, gs)
    bias = np.repeat(mb.astype(np.float64), gs, axis=1)
    assert np.all(np.abs(D - R) <= _U * np.abs(bias) * (1.0 + 1e-12))


def pin_mlx_degenerate(orc):
    """A zero scale (w = bias for every code) and a scale so small that
    -bias/scale overflows are rewritten to codes 1, scale = bias, zero 0, so
    this format's dequant gives the bias exactly (the page's value for the
    overflow group rounds to the bias in binary32); other groups' words pass
    through unchanged."""
    packed, ms, mb, K, N, gs = _mlx_problem(35)
    ms[1, 2] = 0.0
    ms[3, 0] = -0.0
    mb[3, 0] = 0.0
    ms[4, 1] = 1e-38
    mb[4, 1] = 3e38
    Bq, s, z = orc.from_mlx(packed, ms, mb, K, N, gs)
    D = orc.dequant_f64(Bq, s, z, K, N, gs)
    R = orc.mlx_dequant_f64(packed, ms, mb, K, N, gs)
    wpg = gs // 8
    for n, g in ((1, 2), (3, 0), (4, 1)):
        seg = slice(g * gs, (g + 1) * gs)
        assert np.all(D[n, seg] == np.float64(mb[n, g]))
        assert np.all(R[n, seg].astype(np.float32) == mb[n, g])
        assert np.all(Bq[n, g * wpg:(g + 1) * wpg] == 0x11111111)
    keep = np.ones_like(packed, dtype=bool)
    for n, g in ((1, 2), (3, 0), (4, 1)):
        keep[n, g * wpg:(g + 1) * wpg] = False
    assert np.array_equal(Bq[keep], packed[keep])


def pin_embedding_rows(orc):
    """Each gathered row equals an independent numpy binary32 dequant of the
    byte-view codes of that table row, fl(fl(q - z) * s), for repeated,
    first and last ids; an id of -1 or V gives a NaN row and is counted."""
    r = _rng(36)
    V, K, gs = 37, 192, 64
    G = K // gs
    Bq = r.integers(0, 2**32, size=(V, K // 8), dtype=np.uint32)
    s = r.uniform(0.005, 0.02, size=(V, G)).astype(np.float32)
    z = r.uniform(6.0, 9.0, size=(V, G)).astype(np.float32)
    ids = np.array([5, 0, 36, 5, -1, 17, 37, 2], np.int32)
    out, bad = orc.embedding(ids, Bq, s, z, K, gs)
    assert bad == 2
    codes = byte_view_codes(Bq, K, V).astype(np.float32)
    for t, v in enumerate(ids):
        if v < 0 or v >= V:
            assert np.all(np.isnan(out[t]))
            continue
        sv = np.repeat(s[v], gs)
        zv = np.repeat(z[v], gs)
        expect = ((codes[v] - zv).astype(np.float32) * sv).astype(np.float32)
        assert np.array_equal(out[t].view(np.uint32), expect.view(np.uint32))


ALL_PINS = [
    pin_fixed_words, pin_byte_view, pin_pack_round_trip, pin_one_hot, pin_dequant_f32,
    pin_brute_force_exact, pin_abs_sum, pin_zero_point_exact, pin_lanes_independent,
    pin_quad_routing, pin_norm_constant, pin_norm_gain_closed_form, pin_norm_scale_invariance, pin_norm_residual,
    pin_gated_closed_forms, pin_silu_values, pin_gated_norm,
    pin_gated_input_saturation,
    pin_gated_input_values,
    pin_quantize_grid, pin_quantize_nearest, pin_quantize_special_groups,
    pin_mlx_worked_example, pin_mlx_conversion, pin_mlx_degenerate,
    pin_embedding_rows,
]

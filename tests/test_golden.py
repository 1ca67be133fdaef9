"""The oracle against the cited fixtures in tests/golden/ (CPU).

Each fixture names the page passage it follows and how its values were
obtained (the page's own constants, or values evaluated by hand from a
printed formula).
"""

import json
import os
from decimal import Decimal

import numpy as np
import pytest

from int4_group_quantized_quant_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        d = json.load(f)
    assert d["citation"] and d["basis"]
    return d


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.load()


def test_word_layout(orc):
    d = load("int4_word_layout.json")
    for word, codes in d["words"].items():
        Bq = np.array([[int(word, 16)]], np.uint32)
        assert list(orc.unpack(Bq, 8, 1)[0]) == codes, word
    g = d["group_of_vec4u"]
    K, gs = g["K"], g["group_size"]
    # one-hot codes and a distinct scale per group: w(k) names k's group
    G = K // gs
    codes = np.ones((1, K), np.uint8)
    Bq = orc.pack(codes)
    scales = np.arange(1, G + 1, dtype=np.float32).reshape(1, G)
    zeros = np.zeros((1, G), np.float32)
    W = orc.dequant_f64(Bq, scales, zeros, K, 1, gs)[0]
    for v, grp in zip(g["vec4u"], g["group"]):
        assert np.all(W[32 * v:32 * (v + 1)] == grp + 1), (v, grp)


def test_mlx_affine_example(orc):
    d = load("mlx_affine_example.json")
    rows, cols, gs = d["rows"], d["cols"], d["group_size"]
    packed = np.array([[int(w, 16) for w in d["packed"]]], np.uint32)
    ms = np.array([d["scales"]], np.float32)
    mb = np.array([d["biases"]], np.float32)
    expect = np.array(d["expected_w"])
    assert np.array_equal(orc.mlx_dequant_f64(packed, ms, mb, cols, rows, gs)[0], expect)
    Bq, s, z = orc.from_mlx(packed, ms, mb, cols, rows, gs)
    assert z[0, 0] == d["expected_zero"]
    assert np.array_equal(orc.dequant_f64(Bq, s, z, cols, rows, gs)[0], expect)


def test_norm_eps_default(orc):
    d = load("norm_eps_default.json")
    eps = np.float32(d["eps_default"])
    assert hex(int(eps.view(np.uint32))) == d["eps_f32_bits"]
    # the stack's inputs use the page's default
    assert np.float32(I.NORM_EPS) == eps
    c = d["constant_input"]
    K = c["K"]
    A = np.full((1, K), c["value"], np.float32)
    Wn = np.full((K,), c["W_norm"], np.float32)
    _, a, _ = orc.norm(A, None, Wn, eps, K)
    expect = float(Decimal(c["expected_a"]))
    assert np.all(np.abs(a - expect) <= 2e-16 * expect)
    # a gain of distinct powers of two: a_k = c * W_k / sqrt(c^2 + eps)
    g = d["constant_input_gain"]
    K = g["K"]
    A = np.full((1, K), g["value"], np.float32)
    Wn = np.array(g["W_norm"], np.float32)
    _, a, _ = orc.norm(A, None, Wn, eps, K)
    expect = np.array([float(Decimal(v)) for v in g["expected_a"]])
    assert np.all(np.abs(a[0] - expect) <= 2e-16 * np.abs(expect))

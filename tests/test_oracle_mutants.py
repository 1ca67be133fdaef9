"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant is a one-line edit of ``oracle/gq4_oracle.c`` of the kind a
reader could plausibly make (a reversed nibble order, a dropped zero point, a
wrong group index, a dropped term, a wrong sign, ...).  The mutated source is
compiled into a temporary library on the CPU and the pins are run against it.
All mutants keep every memory access in bounds.
"""

import os
import subprocess

import pytest

from tests import oracle_pins as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gq4_oracle.c")

MUTANTS = {
    "nibble_order_reversed": ("(word >> (4 * (k % 8)))", "(word >> (4 * (7 - k % 8)))"),
    "zero_point_sign": ("(q - (double)zeros[g]) * (double)scales[g]",
                        "((double)zeros[g] - q) * (double)scales[g]"),
    "zero_point_dropped": ("(q - (double)zeros[g]) * (double)scales[g]",
                           "q * (double)scales[g]"),
    "scale_dropped": ("(q - (double)zeros[g]) * (double)scales[g]", "(q - (double)zeros[g])"),
    "group_index_wraps": ("(size_t)(k / gs);", "(size_t)(k % (K / gs));"),
    "group_index_off_by_one": ("(size_t)(k / gs);", "(size_t)((k + 1) / gs < K / gs ? (k + 1) / gs : k / gs);"),
    "last_term_dropped": ("for (int k = 0; k < K; ++k) {\n        const double term =\n",
                          "for (int k = 0; k < K - 1; ++k) {\n        const double term =\n"),
    "dot_last_term_dropped": ("for (int k = 0; k < K; ++k) {\n        const double term = a[k]",
                              "for (int k = 0; k < K - 1; ++k) {\n        const double term = a[k]"),
    "abs_sum_signed": ("abs_sum += fabs(term);", "abs_sum += term;"),
    "norm_mean_over_k_minus_1": ("sum_sq / (double)K", "sum_sq / (double)(K - 1)"),
    "norm_eps_dropped": ("sum_sq / (double)K + (double)eps", "sum_sq / (double)K"),
    "norm_residual_second_addend_dropped": ("volatile float xk = ab ? aa[k] + ab[k] : aa[k];\n            if (x)",
                                            "volatile float xk = aa[k];\n            if (x)"),
    "norm_gain_dropped": ("* inv_rms * (double)W_norm[k]", "* inv_rms"),
    "norm_gain_index_off_by_one": ("* inv_rms * (double)W_norm[k]", "* inv_rms * (double)W_norm[(k + 1) % K]"),
    "norm_sqrt_dropped": ("1.0 / sqrt(sum_sq", "1.0 / (sum_sq"),
    "silu_sign": ("t / (1.0 + exp(-t))", "t / (1.0 + exp(t))"),
    "gate_up_swapped": ("out[at] = silu(gv) * uv;", "out[at] = silu(uv) * gv;"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-t));", "return 1.0 / (1.0 + exp(t));"),
    "gated_input_x_g_swapped": ("a[i] = kind == 0 ? x * sigmoid(g) : silu(g) * x;",
                                "a[i] = kind == 0 ? g * sigmoid(x) : silu(x) * g;"),
    "gated_input_kinds_swapped": ("a[i] = kind == 0 ? x * sigmoid(g) : silu(g) * x;",
                                  "a[i] = kind == 1 ? x * sigmoid(g) : silu(g) * x;"),
    "quantize_16_steps": ("volatile float s = d / 15.0f;", "volatile float s = d / 16.0f;"),
    "quantize_zero_sign": ("volatile float z = -lo / s;", "volatile float z = lo / s;"),
    "quantize_floor": ("float qf = rintf(t);", "float qf = floorf(t);"),
    "quantize_min_not_tracked": ("if (v[i] < lo) lo = v[i];", "if (v[i] < lo) hi = hi;"),
    "quantize_nonfinite_unchecked": ("if (!isfinite(v[i])) bad = 1;", "if (!isfinite(v[i])) bad = 0;"),
    "mlx_bias_sign": ("volatile float z = -b / s;", "volatile float z = b / s;"),
    "mlx_degenerate_codes_zero": ("Bq[w0 + j] = 0x11111111u;", "Bq[w0 + j] = 0x00000000u;"),
    "embedding_row_of_position": ("const size_t g = group_index(K, gs, v, k);\n            volatile float d = (float)gq4o_nibble(Bq, K, v, k)",
                                  "const size_t g = group_index(K, gs, t % V, k);\n            volatile float d = (float)gq4o_nibble(Bq, K, t % V, k)"),
    "embedding_last_id_rejected": ("if (v < 0 || v >= V) {", "if (v < 0 || v >= V - 1) {"),
    "embedding_zero_dropped": ("volatile float d = (float)gq4o_nibble(Bq, K, v, k) - zeros[g];",
                               "volatile float d = (float)gq4o_nibble(Bq, K, v, k);"),
    "dequant_f32_double_rounding_skipped": ("volatile float t = (float)gq4o_nibble(Bq, K, n, k) - zeros[g];",
                                            "volatile double t = (double)gq4o_nibble(Bq, K, n, k) - zeros[g];"),
}


# Mutants that a closed form (not a restatement of the oracle's formula) must
# catch: the named pin has to be among the failing ones.
CAUGHT_BY = {
    "norm_gain_dropped": "pin_norm_gain_closed_form",
    "norm_gain_index_off_by_one": "pin_norm_gain_closed_form",
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    import oracle.oracle as O
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutant {name}: pattern not found"
    mutated = source.replace(old, new)
    src = tmp_path / "gq4_oracle.c"
    src.write_text(mutated)
    (tmp_path / "gq4_oracle.h").write_text(open(os.path.join(ROOT, "oracle", "gq4_oracle.h")).read())
    lib = tmp_path / f"libmut_{name}.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(lib), str(src), "-lm"], check=True)
    orc = O.Oracle(O.load_library(str(lib)))
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
    if name in CAUGHT_BY:
        assert CAUGHT_BY[name] in failed, f"mutant {name} not caught by {CAUGHT_BY[name]}: {failed}"

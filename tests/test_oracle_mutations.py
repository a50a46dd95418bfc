"""The oracle's pins catch plausible mistakes.

Each case copies the oracle's C source to a temporary directory, plants one
mistake that a careful reader could still make (a scale taken from the wrong
slab or row, the bias ignored or the biased score used for the gates, equal
scores broken the other way, the wrong divisor in the tile scale, a dropped gate
factor, a flipped sign in a backward term, the bias moved the wrong way),
compiles it into a separate library, loads a separate copy of the oracle's
Python interface on it, and runs the pin that should expose that mistake: the
pin must fail.  The oracle itself is not modified."""
import importlib.util
import os

import pytest

from tests import (test_oracle_backward as tb, test_oracle_dispatch_bias as tdb,
                   test_oracle_gemm as tg, test_oracle_quant as tq, test_oracle_route as tr,
                   test_oracle_wgrad as tw)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_C = os.path.join(ROOT, "oracle", "moe_oracle.c")
ORACLE_PY = os.path.join(ROOT, "oracle", "oracle.py")

# name, text in the oracle, planted text, the pin that must fail, its arguments
MUTATIONS = [
    ("gemm_scale_of_first_slab",
     "sw[(int64_t)(n / 128) * kb_n + kb];", "sw[(int64_t)(n / 128) * kb_n];",
     tg.test_exact_integer_case, {}),
    ("tile_scale_divisor",
     "float scale = amax / 448.0f;", "float scale = amax / 447.0f;",
     tq.test_amax_element_maps_to_448_and_error_bound, {}),
    ("route_bias_ignored",
     "z[i] = s[i] + bias[i];", "z[i] = s[i];",
     tr.test_bias_changes_selection_not_gate_values, {}),
    ("gates_from_biased_scores",
     "gate[(int64_t)t * K + k] = (float)((double)s[idx[(int64_t)t * K + k]] / ssum);",
     "gate[(int64_t)t * K + k] = (float)((double)z[idx[(int64_t)t * K + k]] / ssum);",
     tr.test_bias_changes_selection_not_gate_values, {}),
    ("ties_to_higher_index",
     "if (best < 0 || z[i] > z[best]) best = i;", "if (best < 0 || z[i] >= z[best]) best = i;",
     tr.test_exact_ties_break_by_lower_index_and_flag, {}),
    ("bias_update_reversed",
     "if (load > n) bias[e] = bias[e] - gamma;", "if (load > n) bias[e] = bias[e] + gamma;",
     tdb.test_bias_update_sign_rule, {}),
    ("silu_backward_sign",
     "dgu[i] = dH[i] * U[i] * sgm * (1.0f + G[i] * (1.0f - sgm));",
     "dgu[i] = dH[i] * U[i] * sgm * (1.0f - G[i] * (1.0f - sgm));",
     tb.test_against_float64_chain, {}),
    ("gate_term_sign",
     "const double dl = (dg[k] - gdg) / ssum", "const double dl = (gdg - dg[k]) / ssum",
     tb.test_gate_term_is_there_with_its_sign, {}),
    ("requant_scale_of_first_row",
     "col[i] = v * s[(int64_t)(r0 + i) * (C / 128) + c / 128];",
     "col[i] = v * s[(int64_t)r0 * (C / 128) + c / 128];",
     tw.test_requant_128x1_equals_row_quantiser_on_the_transpose, {}),
    ("wgrad_gate_dropped",
     "dy[(int64_t)r * d + j] = g >= E ? v : gk[r] * v;", "dy[(int64_t)r * d + j] = v;",
     tw.test_layer_wgrad_matches_the_gradient, {"g": 3}),
    ("rowscaled_gemm_wrong_column_scale",
     "float sc = sa[(int64_t)n * kb_n + kb] * sb[(int64_t)m * kb_n + kb];",
     "float sc = sa[(int64_t)n * kb_n + kb] * sb[(int64_t)(m % Na) * kb_n + kb];",
     tw.test_rowscaled_gemm_exact_on_integers, {}),
]


def _mutant(tmp_path, name, old, new):
    src = open(ORACLE_C).read()
    assert src.count(old) >= 1, f"{name}: the text to mutate is not in the oracle"
    d = tmp_path / name
    d.mkdir()
    (d / "moe_oracle.c").write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}", ORACLE_PY)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(d / "moe_oracle.c")
    mod._LIB = str(d / "liboracle.so")
    mod._lib = None
    return mod


@pytest.mark.parametrize("name,old,new,pin,kw", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_planted_mistake(tmp_path, orc, name, old, new, pin, kw):
    pin(orc, **kw)                      # the pin holds on the oracle as it is
    bad = _mutant(tmp_path, name, old, new)
    with pytest.raises(AssertionError):
        pin(bad, **kw)

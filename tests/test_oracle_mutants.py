"""Planted mistakes in a copy of the oracle source must each fail at least one pin.

The mistakes are the plausible ones: a dropped term, a wrong sign, a wrong index, a
transposed operand, a missing rescale. Each mutant is compiled from the committed
source with one textual change, on the CPU; nothing here touches the CUDA path.
"""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    "bias_dropped": ("S_row[j] = p->scale * dot + bias_value(p, bh, i, j);",
                     "S_row[j] = p->scale * dot;"),
    "scale_dropped": ("S_row[j] = p->scale * dot + bias_value(p, bh, i, j);",
                      "S_row[j] = dot + bias_value(p, bh, i, j);"),
    "causal_flipped": ("return j > i ? -INFINITY : 0.0;", "return j < i ? -INFINITY : 0.0;"),
    "causal_diagonal_masked": ("return j > i ? -INFINITY : 0.0;",
                               "return j >= i ? -INFINITY : 0.0;"),
    "key_row_uses_query_index": ("const uint16_t *k = p->K + (bh * N + j) * d;",
                                 "const uint16_t *k = p->K + (bh * N + i) * d;"),
    "value_row_uses_query_index": ("const uint16_t *v = p->V + (bh * N + j) * dv;",
                                   "const uint16_t *v = p->V + (bh * N + i) * dv;"),
    "values_read_from_keys": ("O_row[c] += P_row[j] * bf16_value(v[c]);",
                              "O_row[c] += P_row[j] * bf16_value(p->K[(bh * N + j) * d + c % d]);"),
    "max_not_subtracted_in_sum": ("l += exp(S_row[j] - m);", "l += exp(S_row[j]);"),
    "normalisation_dropped": ("P_row[j] = exp(S_row[j] - m) / l;", "P_row[j] = exp(S_row[j] - m);"),
    "lse_without_log": ("*lse = m + log(l);", "*lse = m + l;"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "bias_row_col_swapped": ("return (double)p->C[(bh * p->N + i) * p->N + j];",
                             "return (double)p->C[(bh * p->N + j) * p->N + i];"),
    "recurrence_alpha_sign": ("double alpha = exp(m - m_new);", "double alpha = exp(m_new - m);"),
    "recurrence_l_not_rescaled": ("l = alpha * l + block_sum;", "l = l + block_sum;"),
    "recurrence_o_not_rescaled": ("o[c] *= alpha;", "o[c] *= 1.0;"),
    "recurrence_running_max_is_block_max": ("double m_new = m > b ? m : b;", "double m_new = b;"),
    "step_r_not_applied_to_l": ("*l = r * *l + p;", "*l = *l + p;"),
    "step_p_relative_to_old_max": ("double p = exp(s - m_new);", "double p = exp(s - *m);"),
    "merge_weights_swapped": ("*l = a1 * l1 + a2 * l2;", "*l = a2 * l1 + a1 * l2;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    pytest.importorskip("mpmath")
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    orc = oracle.Oracle(src.replace(old, new))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, ZeroDivisionError, OverflowError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"

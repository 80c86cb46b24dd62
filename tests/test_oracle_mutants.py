"""Planted mistakes in a copy of the oracle source must each fail at least one pin.

The mistakes are the plausible ones: a dropped term, a wrong sign, a wrong index, a
transposed operand, a missing rescale. Each mutant is compiled from the committed
source with one textual change, on the CPU, and the pins run against it in a child
process (a mutant that reads out of bounds and crashes counts as caught); nothing
here touches the CUDA path.
"""
import os
import subprocess
import sys

import pytest

import oracle

MUTANTS = {
    "bias_dropped": ("        c += (double)p->C[(bh * p->Nq + i) * p->Nk + j];\n", "\n"),
    "scale_dropped": ("S_row[j] = p->scale * dot + bias_value(p, bh, i, j);",
                      "S_row[j] = dot + bias_value(p, bh, i, j);"),
    "all_bias_dropped": ("S_row[j] = p->scale * dot + bias_value(p, bh, i, j);",
                         "S_row[j] = p->scale * dot;"),
    "causal_flipped": ("(p->mode & ORACLE_CAUSAL) && j > i + (p->Nk - p->Nq)",
                       "(p->mode & ORACLE_CAUSAL) && j < i + (p->Nk - p->Nq)"),
    "causal_diagonal_masked": ("(p->mode & ORACLE_CAUSAL) && j > i + (p->Nk - p->Nq)",
                               "(p->mode & ORACLE_CAUSAL) && j >= i + (p->Nk - p->Nq)"),
    "causal_offset_dropped": ("(p->mode & ORACLE_CAUSAL) && j > i + (p->Nk - p->Nq)",
                              "(p->mode & ORACLE_CAUSAL) && j > i"),
    "causal_offset_sign": ("(p->mode & ORACLE_CAUSAL) && j > i + (p->Nk - p->Nq)",
                           "(p->mode & ORACLE_CAUSAL) && j > i + (p->Nq - p->Nk)"),
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
    "bias_row_col_swapped": ("c += (double)p->C[(bh * p->Nq + i) * p->Nk + j];",
                             "c += (double)p->C[(bh * p->Nq + j) * p->Nk + i];"),
    "key_bias_dropped": ("        c += (double)p->ckey[bh * p->Nk + j];\n", "\n"),
    "key_bias_uses_query_index": ("c += (double)p->ckey[bh * p->Nk + j];",
                                  "c += (double)p->ckey[bh * p->Nk + i];"),
    "recurrence_alpha_sign": ("double alpha = exp(m - m_new);", "double alpha = exp(m_new - m);"),
    "recurrence_l_not_rescaled": ("l = alpha * l + block_sum;", "l = l + block_sum;"),
    "recurrence_o_not_rescaled": ("o[c] *= alpha;", "o[c] *= 1.0;"),
    "recurrence_running_max_is_block_max": ("double m_new = m > b ? m : b;", "double m_new = b;"),
    "step_r_not_applied_to_l": ("*l = r * *l + p;", "*l = *l + p;"),
    "step_p_relative_to_old_max": ("double p = exp(s - m_new);", "double p = exp(s - *m);"),
    "merge_weights_swapped": ("*l = a1 * l1 + a2 * l2;", "*l = a2 * l1 + a1 * l2;"),
    "bwd_row_D_dropped": ("const double ds = P_row[j] * (dP_row[j] - D);",
                          "const double ds = P_row[j] * dP_row[j];"),
    "bwd_key_D_dropped": ("const double ds = P * (dP - job->D[i]);", "const double ds = P * dP;"),
    "bwd_D_not_weighted_by_P": ("D += P_row[j] * acc;", "D += acc;"),
    "bwd_dQ_scale_dropped": ("dq[c] *= p->scale;", "dq[c] *= 1.0;"),
    "bwd_dK_scale_dropped": ("dk[c] *= p->scale;", "dk[c] *= 1.0;"),
    "bwd_dK_from_keys": ("dk[c] += ds * bf16_value(q[c]);", "dk[c] += ds * bf16_value(k[c]);"),
    "bwd_dQ_from_queries": ("dq[c] += ds * bf16_value(k[c]);",
                            "dq[c] += ds * bf16_value(p->Q[(bh * p->Nq + i) * d + c]);"),
    "bwd_dV_from_dP": ("dv_out[c] += P * bf16_value(go[c]);", "dv_out[c] += dP * bf16_value(go[c]);"),
    "bwd_key_pass_bias_dropped": ("const double s = p->scale * dot + bias_value(p, bh, i, j);",
                                  "const double s = p->scale * dot;"),
    "bwd_key_pass_unnormalised": ("const double P = exp(s - job->m[i]) / job->l[i];",
                                  "const double P = exp(s - job->m[i]);"),
    "bwd_dP_with_keys": ("acc += bf16_value(go[c]) * bf16_value(v[c]);",
                         "acc += bf16_value(go[c]) * bf16_value(p->K[(bh * Nk + j) * d + c % d]);"),
}

_CHILD = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
orc = oracle.Oracle(open({src!r}).read())
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(orc)
    except Exception as e:  # any failure of a pin counts
        failed.append(pin.__name__)
print("FAILED_PINS", len(failed), ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    pytest.importorskip("mpmath")
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(root=os.path.dirname(tests), tests=tests, src=str(mutant))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return  # the mutant crashed the pins' process: caught
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED_PINS")]
    assert line, r.stdout + r.stderr
    assert int(line[0].split()[1]) > 0, f"mutant {name} passed every pin"

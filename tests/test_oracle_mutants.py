"""The pins must fail on a broken oracle.

Each case plants one plausible mistake in a copy of the oracle's C source,
builds it into a temporary library, and runs the pin suite against it in a
child process: the suite has to fail.  Everything runs on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = {
    "gate_and_up_swapped": ("g += weight_at(L, w13, s13, 2 * I, d, i, c) * h[c];",
                            "g += weight_at(L, w13, s13, 2 * I, d, I + i, c) * h[c];"),
    "down_projection_transposed": ("o += weight_at(L, w2, s2, d, I, r, i) * a[i];",
                                   "o += weight_at(L, w2, s2, I, d, i, r) * a[i];"),
    "scale_block_transposed": ("scale[(size_t)(row / ORC_BLOCK) * scale_cols + col / ORC_BLOCK]",
                               "scale[(size_t)(col / ORC_BLOCK) * scale_cols + row / ORC_BLOCK]"),
    "ties_to_higher_id": ("return (x->id > y->id) - (x->id < y->id);",
                          "return (x->id < y->id) - (x->id > y->id);"),
    "e4m3_bias_8": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);",
                    "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "subnormal_exponent": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "shared_expert_dropped": ("for (int s = 0; s < L->n_shared; ++s)", "for (int s = 0; s < 0; ++s)"),
    "silu_without_gate_factor": ("a[i] = g / (1.0 + exp(-g)) * u;", "a[i] = 1.0 / (1.0 + exp(-g)) * u;"),
    "softmax_not_renormalised": ("for (int j = 0; j < k; ++j) w[j] = exp(z[ids[j]] - zmax) / sum;\n  } else {",
                                 "for (int j = 0; j < k; ++j) w[j] = exp(z[ids[j]] - zmax);\n  } else {"),
    "plan_not_stable": ("for (int p = 0; p < n_slots; ++p)\n      if (ids[p] == uniq[u]) perm[pos++] = p;",
                        "for (int p = n_slots - 1; p >= 0; --p)\n      if (ids[p] == uniq[u]) perm[pos++] = p;"),
    "scale_bytes_dropped": ("*scales = (int64_t)4 *", "*scales = (int64_t)0 *"),
    "budget_keeps_least_contribution": ("return x->score < y->score ? 1 : -1;",
                                        "return x->score > y->score ? 1 : -1;"),
    "budget_ties_to_higher_id": ("return x->id < y->id ? -1 : (x->id > y->id ? 1 : 0);",
                                 "return x->id > y->id ? -1 : (x->id < y->id ? 1 : 0);"),
    "budget_counts_slots_not_weights": ("score[ids[p]] += w[p];", "score[ids[p]] += 1.0;"),
    "budget_one_too_few": ("int kept = U < budget ? U : budget;",
                           "int kept = U < budget ? U : budget - 1;"),
    "budget_dropped_slot_still_summed": ("if (keep && !keep[ids[j]]) continue;",
                                         "if (0 && keep && !keep[ids[j]]) continue;"),
    "budget_dropped_weight_kept": ("w_kept[p] = keep[ids[p]] ? w[p] : 0.0;", "w_kept[p] = w[p];"),
    "budget_plan_counts_dropped": ("if (keep[ids[p]]) hist[ids[p]] += 1;", "hist[ids[p]] += 1;"),
    "tree_score_skips_own_factor": ("for (int i = len - 1; i >= 0; --i) s *= (double)q[path[i]];",
                                    "for (int i = len - 1; i >= 1; --i) s *= (double)q[path[i]];"),
    "evict_ties_to_higher_index": ("return (x->v > y->v) - (x->v < y->v);",
                                   "return (x->v < y->v) - (x->v > y->v);"),
    "evict_argmax_last_on_tie": ("if (utility[k - 1] > utility[best - 1]) best = k;",
                                 "if (utility[k - 1] >= utility[best - 1]) best = k;"),
    "evict_cost_index_shifted": ("utility[k - 1] = acc / (double)cost[k - 1];",
                                 "utility[k - 1] = acc / (double)cost[k > 1 ? k - 2 : 0];"),
    "ecospec_cost_ignores_buffer": ("cost += tv[i] && !buf_out[i];", "cost += tv[i];"),
    "ecospec_buffer_not_updated": ("for (size_t i = 0; i < LE; ++i) buf_out[i] |= tb[i];",
                                   "for (size_t i = 0; i < LE; ++i) buf_out[i] |= 0 * tb[i];"),
    "ecospec_path_without_ancestors": ("      if (u == 0) break;\n    }", "      if (1) break;\n    }"),
    "ecospec_eps_ignored": ("const double score = P[v] / ((double)cost + eps);",
                            "const double score = P[v] / ((double)cost + 1.0);"),
    "ecospec_ties_to_higher_index": ("if (best < 0 || score > best_score) {",
                                     "if (best < 0 || score >= best_score) {"),
    "given_routing_gated_on_top_k": ("  orc_router_scores(L, h, z);\n  orc_gate(z, L->n_experts, ids, L->top_k, L->gate, w);\n  free(h);\n}\n\n/* The layer output",
                                     "  orc_router_scores(L, h, z);\n  orc_topk(z, L->n_experts, L->top_k, (int32_t *)ids);\n  orc_gate(z, L->n_experts, ids, L->top_k, L->gate, w);\n  free(h);\n}\n\n/* The layer output"),
    "budget_plan_not_stable": ("for (int p = 0; p < n_slots; ++p)\n      if (uniq[u] == ids[p])",
                               "for (int p = n_slots - 1; p >= 0; --p)\n      if (uniq[u] == ids[p])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", str(lib), str(mut), "-lm"])
    env = dict(os.environ, MOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins passed on mutant {name}:\n{r.stdout[-2000:]}"

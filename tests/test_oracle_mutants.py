"""Planted mistakes in the oracle must trip its pins (CPU only).

Each case copies ``oracle/spec_verify_oracle.c``, makes one plausible mistake
(a dropped term, a wrong sign, index or lane, a swapped operand, a loosened
check), compiles the copy and runs the pins of ``oracle_pins`` against it.
At least one pin has to fail, which shows that the pins constrain every part
of the oracle rather than restating it.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spec_verify_oracle.c")

MUTANTS = {
    "residual_without_clamp": ("r[x] = d > 0.0 ? d : 0.0;", "r[x] = d;"),
    "ratio_inverted": ("u <= px / qx", "u <= qx / px"),
    "temperature_dropped": ("p[x] = exp(l[x] / T - M);", "p[x] = exp(l[x] - M);"),
    "no_break_after_rejection": (
        "emitted = inverse_cdf(p, V, u_emit[j], &mass, &lo, &hi, probe, &plo, &phi);\n"
        "        }\n        break;",
        "emitted = inverse_cdf(p, V, u_emit[j], &mass, &lo, &hi, probe, &plo, &phi);\n"
        "        }\n        continue;"),
    "inverse_cdf_strict": ("if (pick < 0 && C >= t)", "if (pick < 0 && C > t)"),
    "argmax_last_tie": ("if (l[x] > l[best]) best = x;", "if (l[x] >= l[best]) best = x;"),
    "uniform_lanes_swapped": ("*u_accept = oracle_uniform_from_bits(out[0]);",
                              "*u_accept = oracle_uniform_from_bits(out[1]);"),
    "philox_wrong_product": ("uint32_t n0 = hi1 ^ c1 ^ k0;", "uint32_t n0 = hi0 ^ c1 ^ k0;"),
    "philox_no_key_schedule": ("k0 += PHILOX_WEYL0;", "k0 += 0u;"),
    "uniform_includes_zero": ("return (double)((x >> 8) + 1u) * (1.0 / 16777216.0);",
                              "return (double)(x >> 8) * (1.0 / 16777216.0);"),
    "softmax_unnormalised": ("for (int x = 0; x < V; ++x) p[x] /= Z;", "(void)Z;"),
    "bonus_from_previous_row": ("load_logit_row(logits, dtype, K, V, b, n, l);\n        erow = n;",
                                "load_logit_row(logits, dtype, K, V, b, n - (n > 0), l);\n"
                                "        erow = n;"),
    "residual_sign_flipped": ("double d = p[x] - (double)q[x];", "double d = (double)q[x] - p[x];"),
    "zero_target_guard_dropped": ("(px > 0.0) && (qx == 0.0 ||", "(qx == 0.0 ||"),
    "emission_reuses_acceptance_uniform": ("emitted = inverse_cdf(r, V, u_emit[j],",
                                           "emitted = inverse_cdf(r, V, u_accept[j],"),
    "emitted_at_wrong_slot": ("out_ids[accepted] = emitted;", "out_ids[n] = emitted;"),
    "greedy_emits_draft": ("emitted = g; /* the target's own token replaces the mismatch */",
                           "emitted = xj;"),
    "negative_temperature_allowed": ("if (!(T >= 0.0) || isinf(T)) return -1;",
                                     "if (isnan(T) || isinf(T)) return -1;"),
    "empty_row_not_rejected": ("if (!finite) return -1;", "(void)finite;"),
    "typical_threshold_strict": ("(px >= threshold)", "(px > threshold)"),
    "typical_zero_guard_dropped": ("(px > 0.0) && (px >= threshold)", "(px >= threshold)"),
    "typical_emission_uses_acceptance_uniform": (
        "mode = 4;\n            emitted = inverse_cdf(p, V, u_emit[j],",
        "mode = 4;\n            emitted = inverse_cdf(p, V, u_accept[j],"),
    "tree_residual_not_renormalised": ("for (int y = 0; y < V; ++y) r[y] = w[y] / S;",
                                       "for (int y = 0; y < V; ++y) r[y] = w[y];"),
    "tree_child_uniform_shifted": ("if (v + 1 < 64) ua[v + 1] = a0;", "if (v < 64) ua[v] = a0;"),
    "tree_greedy_last_matching_child": ("for (int c = v + 1; c < n && next < 0; ++c)",
                                        "for (int c = v + 1; c < n; ++c)"),
    "tree_emits_from_running_target": ("emit_w = w; /* unnormalised", "emit_w = r; /* unnormalised"),
    "tree_parent_order_unchecked": ("if (par[c] < 0 || par[c] >= c) return -1;",
                                    "if (par[c] < 0) return -1;"),
    "typical_emits_from_next_row": (
        "erow = j;  /* the target's own token at the first refused position */",
        "erow = j;\n            if (j + 1 <= n) load_logit_row(logits, dtype, K, V, b, j + 1, l),"
        " softmax_t(l, V, T, p);"),
}

# cheap pins first, so that most mutants are caught quickly
ORDER = ["pin_philox_kat", "pin_uniform_map", "pin_uniform_lanes", "pin_greedy_example",
         "pin_greedy_ties", "pin_inverse_cdf_ends", "pin_zero_residual_fallback",
         "pin_bad_inputs", "pin_zero_target_prob_never_accepted", "pin_output_shape",
         "pin_softmax_vs_scipy", "pin_temperature", "pin_residual_support",
         "pin_unused_rows_ignored", "pin_request_index", "pin_equal_probs_always_accept",
         "pin_brute_force", "pin_worked_ratio", "pin_lossless_closed_form",
         "pin_typical_threshold_boundary", "pin_typical_brute_force",
         "pin_typical_closed_form", "pin_tree_bad_inputs", "pin_tree_unused_nodes_ignored",
         "pin_tree_chain_is_chain", "pin_tree_brute_force", "pin_tree_first_token_law"]


def test_order_covers_all_pins():
    assert sorted(ORDER) == sorted(p.__name__ for p in oracle_pins.PINS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site of {name} not unique"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(old, new))
    so = oracle.build(str(path), out=str(tmp_path / f"lib_{name}.so"))
    lib = oracle.load(so)
    pins = {p.__name__: p for p in oracle_pins.PINS}
    for pin_name in ORDER:
        try:
            pins[pin_name](lib)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            return  # caught
    pytest.fail(f"no pin caught the planted mistake {name}")

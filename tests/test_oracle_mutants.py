"""Plausible mistakes planted in copies of the oracle must each fail a pin.

Each mutant is the oracle source with one exact text substitution, compiled
with gcc into a temporary directory.  This shows the pins in oracle_pins.py
are strong enough to catch a dropped term, a wrong sign, a wrong index or a
transposed operand.  Everything here runs on the CPU.
"""
import os

import numpy as np
import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spec_verify_ref.c")

MUTANTS = {
    "ratio_inverted": ("const double ratio = (q == 0.0) ? INFINITY : p / q;",
                       "const double ratio = (q == 0.0) ? INFINITY : q / p;"),
    "accept_non_strict": ("(u[i] < ratio)", "(u[i] <= ratio)"),
    "residual_no_clamp": ("r[v] = d > 0.0 ? d : 0.0;", "r[v] = d > 0.0 ? d : -d;"),
    "residual_reversed": ("const double d = p[v] - q[v];", "const double d = q[v] - p[v];"),
    "cdf_non_strict": ("if (c > target) {", "if (c >= target) {"),
    "cdf_unnormalised": ("double target = u * S;", "double target = u;"),
    "resample_reuses_accept_uniform": ("out[k] = inverse_cdf(r, V, S, u[G], &margin);",
                                       "out[k] = inverse_cdf(r, V, S, u[k], &margin);"),
    "bonus_from_first_row": (
        "softmax_row(a->target, a->dtype, target_row(b, k, G, V), V, T, p, &m, &s);",
        "softmax_row(a->target, a->dtype, target_row(b, k < gb ? k : 0, G, V), V, T, p, &m, &s);"),
    "residual_next_draft_row": (
        "softmax_row(a->draft, a->dtype, draft_row(b, k, G, V), V, T, q, &m, &s);",
        "softmax_row(a->draft, a->dtype, draft_row(b, k + 1 < gb ? k + 1 : k, G, V), V, T, q, &m, &s);"),
    "no_bonus_token": ("  out[k] = inverse_cdf(r, V, S, u[G], &margin);",
                       "  out[k] = (k < gb) ? inverse_cdf(r, V, S, u[G], &margin) : -1;"),
    "draft_without_temperature": (
        "const double q = prob_of(a->draft, a->dtype, draft_row(b, i, G, V), x, T, md, sd);",
        "const double q = prob_of(a->draft, a->dtype, draft_row(b, i, G, V), x, 1.0, md, sd);"),
    "softmax_max_sign": ("double e = exp((logit_at(base, dtype, off + (size_t)v) - m) / T);",
                         "double e = exp((m - logit_at(base, dtype, off + (size_t)v)) / T);"),
    "softmax_unnormalised": ("    for (int v = 0; v < V; ++v) p_out[v] /= s;",
                             "    for (int v = 0; v < V; ++v) p_out[v] /= 1.0;"),
    "temperature_multiplies": ("return exp((logit_at(base, dtype, off + (size_t)x) - m) / T) / s;",
                               "return exp((logit_at(base, dtype, off + (size_t)x) - m) * T) / s;"),
    "greedy_tie_highest": ("      } else if (z == zbest) {\n        ties = 1;",
                           "      } else if (z == zbest) {\n        ties = 1; best = v;"),
    "greedy_accepts_mismatch": ("tokens[(size_t)b * G + i] != best",
                                "tokens[(size_t)b * G + i] == best + V"),
    "truncation_keeps_rejected_draft": ("      k = i;\n      break;",
                                        "      k = i + 1;\n      out[i] = x;\n      break;"),
    "vanished_residual_no_fallback": ("    if (S == 0.0) { /* residual vanished: fall back to p */",
                                      "    if (S < 0.0) { /* residual vanished: fall back to p */"),
    "vanished_residual_falls_back_to_q": (
        "    free(q);\n    if (a->resid_mass) a->resid_mass[b] = S;\n"
        "    if (S == 0.0) { /* residual vanished: fall back to p */\n"
        "      for (int v = 0; v < V; ++v) {\n        r[v] = p[v];",
        "    if (a->resid_mass) a->resid_mass[b] = S;\n"
        "    if (S == 0.0) { /* residual vanished: fall back to p */\n"
        "      for (int v = 0; v < V; ++v) {\n        r[v] = q[v];"),
    "vanished_residual_falls_back_to_argmax": (
        "      for (int v = 0; v < V; ++v) {\n        r[v] = p[v];\n        S += r[v];\n      }\n    }\n  } else {",
        "      int am = 0;\n      for (int v = 1; v < V; ++v) if (p[v] > p[am]) am = v;\n"
        "      for (int v = 0; v < V; ++v) {\n        r[v] = v == am ? 1.0 : 0.0;\n        S += r[v];\n"
        "      }\n    }\n  } else {"),
    "cdf_rounding_takes_first_positive": ("  for (int j = V - 1; j >= 0; --j) {\n    if (r[j] > 0.0) {",
                                          "  for (int j = 0; j < V; ++j) {\n    if (r[j] > 0.0) {"),
    "cdf_rounding_takes_last_token": ("  for (int j = V - 1; j >= 0; --j) {\n    if (r[j] > 0.0) {",
                                      "  for (int j = V - 1; j >= 0; --j) {\n    if (j == V - 1) {"),
    "cdf_rounding_takes_largest_weight": (
        "  for (int j = V - 1; j >= 0; --j) {\n    if (r[j] > 0.0) {\n      *margin = 0.0;\n      return j;",
        "  for (int j = V - 1; j >= 0; --j) {\n    if (r[j] > 0.0) {\n      int am = 0;\n"
        "      for (int i = 1; i < V; ++i) if (r[i] > r[am]) am = i;\n      *margin = 0.0;\n      return am;"),
}


def _quick_pins(o):
    """Run the pins in order; return the name of the first that fails."""
    cases = pins.lossless_cases()
    checks = [
        ("lossless_gamma1", lambda: pins.check_lossless_gamma1(o, cases[1])),
        ("lossless_gamma1_T", lambda: pins.check_lossless_gamma1(o, cases[5])),
        ("lossless_gamma2", lambda: pins.check_lossless_gamma2(o, cases[0])),
        ("accept_strict", lambda: pins.check_accept_strict(o)),
        ("inverse_cdf_boundaries", lambda: pins.check_inverse_cdf_boundaries(o)),
        ("vanished_residual", lambda: pins.check_vanished_residual_falls_back_to_p(o)),
        ("subnormal_residual", lambda: pins.check_subnormal_residual_draw(o)),
        ("gamma0", lambda: pins.check_gamma0_bonus_only(o)),
        ("softmax", lambda: pins.check_softmax(o)),
        ("p_q_at_tokens", lambda: pins.check_p_q_at_tokens(o)),
        ("truncation", lambda: pins.check_truncation_and_padding(o)),
        ("expected_tokens", lambda: pins.check_expected_tokens(o, 3, trials=100_000)),
        ("greedy_same_rows", lambda: pins.check_greedy_same_rows(o)),
        ("greedy_worked_example", lambda: pins.check_greedy_worked_example(o)),
        ("greedy_ties", lambda: pins.check_greedy_ties(o)),
    ]
    for name, fn in checks:
        try:
            fn()
        except (AssertionError, ValueError) as e:  # noqa: PERF203
            return name, e
    return None, None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    caught, err = _quick_pins(oracle.Oracle(lib))
    assert caught is not None, f"mutant {name} passed every pin"


def test_real_oracle_passes_quick_pins():
    caught, err = _quick_pins(oracle.default())
    assert caught is None, (caught, err)

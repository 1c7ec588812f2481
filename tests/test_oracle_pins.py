"""The float64 oracle, pinned to what the pages and the mathematics fix (CPU)."""
import json
import os

import numpy as np
import pytest

import oracle
import oracle_pins as pins

ORACLE = oracle.default()


@pytest.mark.parametrize("case", range(len(pins.lossless_cases())))
def test_lossless_enumeration_gamma1(case):
    pins.check_lossless_gamma1(ORACLE, pins.lossless_cases()[case])


@pytest.mark.parametrize("case", [0, 3, 4])
def test_lossless_enumeration_gamma2(case):
    rows = pins.lossless_cases()[case]
    pins.check_lossless_gamma2(ORACLE, rows)


@pytest.mark.parametrize("gamma", [1, 3, 5])
def test_expected_tokens_closed_form(gamma):
    alpha, mean, expect = pins.check_expected_tokens(ORACLE, gamma)
    assert abs(alpha - 0.7) < 1e-6


def test_expected_tokens_printed_values():
    """The closed form reproduces the numbers the pages print (golden file)."""
    g = json.load(open(os.path.join(pins.GOLDEN, "expected_tokens.json")))
    for c in g["cases"]:
        a, k = c["alpha"], c["gamma"]
        e = (1 - a ** (k + 1)) / (1 - a)
        assert round(e, c["decimals"]) == c["printed"], (c, e)
    t = g["terms"]
    terms = [t["alpha"] ** i for i in range(t["gamma"] + 1)]
    for v, printed, dec in zip(terms, t["printed"], t["decimals"]):
        assert round(v, dec) == printed


def test_q_equals_p_accepts_all():
    pins.check_q_equals_p_accepts_all(ORACLE)


def test_disjoint_support_rejects_all():
    pins.check_disjoint_rejects_all(ORACLE)


def test_greedy_same_rows_accepts_all():
    pins.check_greedy_same_rows(ORACLE)


def test_greedy_worked_example():
    pins.check_greedy_worked_example(ORACLE)


def test_greedy_ties_lowest_id():
    pins.check_greedy_ties(ORACLE)


def test_inverse_cdf_boundaries():
    pins.check_inverse_cdf_boundaries(ORACLE)


def test_vanished_residual_falls_back_to_p():
    pins.check_vanished_residual_falls_back_to_p(ORACLE)


def test_subnormal_residual_draw():
    pins.check_subnormal_residual_draw(ORACLE)


def test_gamma0_bonus_only():
    pins.check_gamma0_bonus_only(ORACLE)


def test_masked_tokens():
    pins.check_masked_tokens(ORACLE)


def test_softmax_closed_forms_and_scipy():
    pins.check_softmax(ORACLE)


def test_p_q_at_tokens_match_scipy():
    pins.check_p_q_at_tokens(ORACLE)


def test_truncation_and_padding():
    pins.check_truncation_and_padding(ORACLE)


def test_invalid_input_rejected():
    t = np.zeros((1, 2, 4), np.float32)
    d = np.zeros((1, 1, 4), np.float32)
    ok = dict(draft_tokens=np.array([[1]], np.int32), gamma=np.array([1], np.int32),
              uniforms=np.array([[0.5, 0.5]]), temperature=np.array([1.0], np.float32))
    ORACLE.sample(t, d, **ok)
    for key, bad in (("draft_tokens", np.array([[4]], np.int32)),
                     ("gamma", np.array([2], np.int32)),
                     ("uniforms", np.array([[1.0, 0.5]])),
                     ("temperature", np.array([-1.0], np.float32)),
                     ("temperature", np.array([np.inf], np.float32))):
        args = dict(ok)
        args[key] = bad
        with pytest.raises(ValueError):
            ORACLE.sample(t, d, **args)


def test_zero_temperature_request_takes_the_greedy_steps():
    """A request with T = 0 in a sampling call is verified by argmax matching
    (the explainer's implementation points: temperature -> 0 is greedy), the
    same as the greedy call on that request; the others are unaffected."""
    rng = np.random.default_rng(21)
    B, G, V = 6, 3, 50
    t = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    d = (t[:, :G] + rng.normal(0, 0.5, (B, G, V))).astype(np.float32)
    gamma = np.array([3, 2, 3, 0, 1, 3], np.int32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    x[0] = t[0, :G].argmax(axis=1)           # request 0: every draft is the argmax
    for b in range(B):
        x[b, gamma[b]:] = 0
    u = rng.random((B, G + 1))
    T = np.array([0.0, 0.7, 0.0, 0.0, 1.0, 0.0], np.float32)
    mixed = ORACLE.sample(t, d, x, gamma, u, T)
    greedy = ORACLE.greedy(t, x, gamma)
    sampled = ORACLE.sample(t, d, x, gamma, u, np.where(T == 0, 1.0, T).astype(np.float32))
    for b in range(B):
        ref = greedy if T[b] == 0 else sampled
        assert (mixed["out_tokens"][b] == ref["out_tokens"][b]).all()
        assert mixed["num_accepted"][b] == ref["num_accepted"][b]
        if T[b] == 0:
            assert np.isnan(mixed["p_tok"][b]).all() and np.isnan(mixed["q_tok"][b]).all()
    assert mixed["num_accepted"][0] == 3 and mixed["out_tokens"][0][3] == t[0, 3].argmax()


def test_threads_do_not_change_results():
    rng = np.random.default_rng(12)
    B, G, V = 50, 3, 300
    t = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    d = (t[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    g = rng.integers(0, G + 1, B).astype(np.int32)
    u = rng.random((B, G + 1)).astype(np.float32)
    T = np.ones(B, np.float32)
    a = ORACLE.sample(t, d, x, g, u, T, nthreads=1)
    b = ORACLE.sample(t, d, x, g, u, T, nthreads=4)
    for k in ("out_tokens", "num_accepted"):
        assert np.array_equal(a[k], b[k])


def test_rows_first_gives_identical_results():
    """rows_first only spreads the row statistics over threads first: every
    output (tokens, counts, probabilities, margins, residual mass) is
    bit-identical, including zero-temperature requests and gamma_b = 0."""
    rng = np.random.default_rng(13)
    B, G, V = 7, 4, 333
    t = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    d = (t[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    g = np.array([4, 0, 2, 4, 1, 3, 4], np.int32)
    u = rng.random((B, G + 1)).astype(np.float32)
    T = np.array([1.0, 0.5, 0.0, 1.5, 1.0, 0.8, 1.2], np.float32)
    a = ORACLE.sample(t, d, x, g, u, T, nthreads=1)
    b = ORACLE.sample(t, d, x, g, u, T, nthreads=8, rows_first=True)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k

"""Host-side draft-length policies and the gamma* optimiser, pinned to the
pages' printed values and to simulations that do not use the closed forms."""
import numpy as np
import pytest

from speculative_decoding_verification_62_gb300 import policies as pol


def simulate_tokens(alpha, gamma, steps, rng):
    """Tokens per verify by direct simulation of independent acceptances."""
    acc = rng.random((steps, gamma)) < alpha
    first_reject = np.where(acc.all(axis=1), gamma, np.argmin(acc, axis=1))
    return first_reject + 1


def test_expected_tokens_printed_values():
    # "Speculative Decoding theory": alpha = 0.7, gamma = 5 gives about 2.94;
    # "draft length by load": alpha = 0.7, K = 3 about 2.5, K = 1 1.7.
    assert round(pol.expected_tokens(0.7, 5), 2) == 2.94
    assert round(pol.expected_tokens(0.7, 3), 1) == 2.5
    assert round(pol.expected_tokens(0.7, 1), 1) == 1.7
    assert pol.expected_tokens(0.0, 6) == 1.0
    assert pol.expected_tokens(1.0, 6) == 7.0


def test_expected_tokens_matches_simulation():
    rng = np.random.default_rng(5)
    for a, g in ((0.3, 2), (0.7, 5), (0.9, 7)):
        t = simulate_tokens(a, g, 200_000, rng)
        se = t.std() / np.sqrt(t.size)
        assert abs(t.mean() - pol.expected_tokens(a, g)) < 5 * se


def test_speedup_printed_bound():
    # explainer: c = 0.05, gamma = 5, alpha = 1 -> 6 / 1.25 = 4.8
    assert pol.speedup(1.0, 5, 0.05) == pytest.approx(4.8, rel=1e-15)


def test_optimal_gamma_edges_and_monotonicity():
    assert pol.optimal_gamma(0.0, 0.1) == 0          # every draft rejected: do not draft
    assert pol.optimal_gamma(1.0, 0.1, gamma_max=12) == 12
    alphas = np.linspace(0.0, 0.99, 45)
    gs = [pol.optimal_gamma(a, 0.1) for a in alphas]
    assert all(x <= y for x, y in zip(gs, gs[1:]))   # longer drafts as alpha grows
    cs = np.linspace(0.01, 0.8, 30)
    gc = [pol.optimal_gamma(0.8, c) for c in cs]
    assert all(x >= y for x, y in zip(gc, gc[1:]))   # shorter drafts as drafting costs more


def test_optimal_gamma_agrees_with_simulated_speedup():
    rng = np.random.default_rng(11)
    for a, c in ((0.6, 0.1), (0.8, 0.05), (0.9, 0.2)):
        sim = [simulate_tokens(a, g, 200_000, rng).mean() / (c * g + 1) if g else 1.0
               for g in range(0, 13)]
        best = int(np.argmax(sim))
        g_star = pol.optimal_gamma(a, c, gamma_max=12)
        # the simulated optimum is within noise of the closed-form one
        assert sim[g_star] >= sim[best] * (1 - 0.01)


def test_acceptance_estimator_counts_and_convergence():
    est = pol.AcceptanceEstimator()
    est.update([3, 3], [3, 1])        # 3 + 1 successes, 0 + 1 failures
    assert est.alpha == pytest.approx(4 / 5)
    rng = np.random.default_rng(3)
    est = pol.AcceptanceEstimator()
    for _ in range(50):
        k = simulate_tokens(0.6, 4, 400, rng) - 1
        est.update([4] * k.size, k)
    assert abs(est.alpha - 0.6) < 0.01
    with pytest.raises(ValueError):
        est.update([2], [3])
    decayed = pol.AcceptanceEstimator(decay=0.5)
    decayed.update(4, 4)
    decayed.update(4, 0)
    assert decayed.alpha == pytest.approx(2 / 3)     # 0.5*4 successes, 1 failure


def test_batch_size_table_docs_example():
    t = pol.BatchSizeTable.docs_example()
    assert [t(n) for n in (1, 64, 65, 128, 129, 512, 513)] == [3, 3, 1, 1, 0, 0, 0]
    with pytest.raises(ValueError):
        pol.BatchSizeTable({(1, 64): 3, (60, 128): 1})


def test_accept_length_ema():
    p = pol.AcceptLengthEMA(weight=1.0)
    assert p.steps(32) == 1 and p.steps(200) == 1    # fixed at one step from 32 requests
    assert p.steps(4) == 7                           # no observation yet: the longest candidate
    p.observe(4, [6, 7, 6, 6])                       # mean 6.25 -> round + 1 = 7
    assert p.steps(4) == 7
    p.observe(4, [2, 3, 2, 2.68])                    # mean 2.42 -> 3
    assert p.steps(4) == 3
    p.observe(4, [0, 0])                             # round(0) + 1 = 1, the shortest candidate
    assert p.steps(4) == 1
    q = pol.AcceptLengthEMA(weight=0.5)
    q.observe(2, [4])
    q.observe(2, [0])
    assert q.ema[q._range(2)] == pytest.approx(2.0)
    assert q.steps(2) == 3

"""Checks that pin the float64 oracle to what the pages and the mathematics fix.

Each check takes an ``oracle.Oracle`` instance and raises AssertionError when the
oracle disagrees.  ``test_oracle_pins.py`` runs them on the real oracle (all
must pass); ``test_oracle_mutants.py`` runs them on deliberately broken copies
(at least one must fail for every mutant).

Nothing here restates the oracle's formulas.  The independent references are:
the lossless theorem (emitted marginal equals p), the closed form for the
expected tokens per step, scipy's softmax, exact special cases, and
hand-computed inverse-CDF boundaries.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import softmax as scipy_softmax

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ONE_MINUS = np.nextafter(1.0, 0.0)


# --------------------------------------------------------------------------
# Black-box boundary search over the oracle's double-precision uniforms
# --------------------------------------------------------------------------
def first_true(pred, n):
    """Smallest double u in [0, 1) with pred(u)[j] true, per probe j; 1.0 if none.

    pred maps an array of n doubles to n booleans and must be monotone
    (false then true) in u.  Bisection runs on the IEEE bit patterns, which
    order non-negative doubles, so the result is exact to the last bit.
    """
    lo = np.zeros(n, dtype=np.uint64)                       # candidate answer >= lo
    hi = np.full(n, np.float64(1.0).view(np.uint64), dtype=np.uint64)  # pred(hi) := true
    while np.any(lo < hi):
        active = lo < hi
        mid = np.where(active, lo + (hi - lo) // np.uint64(2), np.uint64(0))
        val = pred(mid.view(np.float64).copy())
        hi = np.where(active & val, mid, hi)
        lo = np.where(active & ~val, mid + np.uint64(1), lo)
    return lo.view(np.float64).copy()


class Rows:
    """One request's rows (float32 logits) replicated into probe batches."""

    def __init__(self, target, draft, T):
        self.t = np.asarray(target, np.float32)   # [G+1][V]
        self.d = np.asarray(draft, np.float32)    # [G][V]
        self.T = np.float32(T)
        self.G = self.t.shape[0] - 1
        self.V = self.t.shape[1]

    def first(self, G):
        """The same request cut to its first G positions."""
        return Rows(self.t[:G + 1], self.d[:G], self.T)

    def run(self, oracle, tokens, u):
        """tokens [n][G], u [n][G+1] (doubles) -> oracle result dict."""
        n = len(u)
        t = np.broadcast_to(self.t, (n,) + self.t.shape).copy()
        d = np.broadcast_to(self.d, (n,) + self.d.shape).copy()
        g = np.full(n, self.G, np.int32)
        T = np.full(n, self.T, np.float32)
        return oracle.sample(t, d, np.asarray(tokens, np.int32).reshape(n, self.G), g,
                             np.asarray(u, np.float64), T)

    def p(self, i):
        return scipy_softmax(self.t[i].astype(np.float64) / np.float64(self.T))

    def q(self, i):
        return scipy_softmax(self.d[i].astype(np.float64) / np.float64(self.T))


def _accept_measure(oracle, rows, tokens, pos, base_u):
    """P(accept at pos) for each probe, found as the reject threshold in u[pos]."""
    n = len(tokens)

    def rejects(u):
        uu = base_u.copy()
        uu[:, pos] = u
        r = rows.run(oracle, tokens, uu)
        return r["num_accepted"] <= pos

    return first_true(rejects, n)


def _cdf_measure(oracle, rows, tokens, base_u, out_pos, expect_nacc):
    """Measure of u_s giving each output token at out_pos: [n][V]."""
    n, V, G = len(tokens), rows.V, rows.G
    edges = np.zeros((n, V + 1))
    edges[:, V] = 1.0
    for y in range(V):
        def beyond(u, y=y):
            uu = base_u.copy()
            uu[:, G] = u
            r = rows.run(oracle, tokens, uu)
            assert np.all(r["num_accepted"] == expect_nacc), "branch changed while probing u_s"
            return r["out_tokens"][:, out_pos] > y
        edges[:, y + 1] = first_true(beyond, n)
    meas = np.diff(edges, axis=1)
    assert np.all(meas >= -1e-15), "inverse CDF is not monotone in u"
    return meas


def check_lossless_gamma1(oracle, rows):
    """gamma = 1: exact enumeration over the draft token and the uniforms.

    The theorem (disassemble-channel 'Speculative Decoding', section 'Proof that
    the output equals the target distribution'): the emitted token has law p;
    split by branch, P(reject, emit y) = max(0, p(y) - q(y)) and
    P(accept x, then bonus y') = min(p(x), q(x)) * p_1(y').
    """
    rows = rows.first(1)
    V = rows.V
    p0, q0, p1 = rows.p(0), rows.q(0), rows.p(1)
    tokens = np.arange(V).reshape(V, 1)
    base = np.zeros((V, 2))
    acc = _accept_measure(oracle, rows, tokens, 0, base)          # [V]
    rej_u = base.copy(); rej_u[:, 0] = ONE_MINUS
    rej_meas = _cdf_measure(oracle, rows, tokens, rej_u, 0, np.where(acc < 1.0, 0, 1))
    acc_u = base.copy(); acc_u[:, 0] = 0.0
    bonus = _cdf_measure(oracle, rows, tokens, acc_u, 1, 1)
    reject_emit = np.zeros(V)
    joint = np.zeros((V, V))
    for x in range(V):
        if acc[x] < 1.0:
            reject_emit += q0[x] * (1.0 - acc[x]) * rej_meas[x]
        joint[x] += q0[x] * acc[x] * bonus[x]
    assert np.allclose(reject_emit, np.maximum(0.0, p0 - q0), rtol=0, atol=1e-12), \
        (reject_emit, np.maximum(0, p0 - q0))
    assert np.allclose(joint, np.minimum(p0, q0)[:, None] * p1[None, :], rtol=0, atol=1e-12)
    first = reject_emit + joint.sum(axis=1)
    assert np.allclose(first, p0, rtol=0, atol=1e-12), (first, p0)


def check_lossless_gamma2(oracle, rows):
    """gamma = 2: exact enumeration over both draft tokens and all uniforms.

    Same theorem applied position by position: P(reject at 0, y) =
    max(0, p0-q0)(y); P(accept y, reject at 1, y') = min(p0,q0)(y) *
    max(0, p1-q1)(y'); P(accept y, y', bonus y'') = min(p0,q0)(y) *
    min(p1,q1)(y') * p2(y'').
    """
    rows = rows.first(2)
    V = rows.V
    p0, q0, p1, q1, p2 = rows.p(0), rows.q(0), rows.p(1), rows.q(1), rows.p(2)
    xs = np.array([(a, b) for a in range(V) for b in range(V)], np.int32)
    n = len(xs)
    w = q0[xs[:, 0]] * q1[xs[:, 1]]
    base = np.zeros((n, 3))
    a0 = _accept_measure(oracle, rows, xs, 0, base)
    a1 = _accept_measure(oracle, rows, xs, 1, base)     # u0 = 0: position 0 accepted
    u_rej0 = base.copy(); u_rej0[:, 0] = ONE_MINUS
    m_rej0 = _cdf_measure(oracle, rows, xs, u_rej0, 0, np.where(a0 < 1.0, 0, 2))
    u_rej1 = base.copy(); u_rej1[:, 1] = ONE_MINUS
    m_rej1 = _cdf_measure(oracle, rows, xs, u_rej1, 1, np.where(a1 < 1.0, 1, 2))
    m_all = _cdf_measure(oracle, rows, xs, base, 2, 2)
    P0 = np.zeros(V)
    P1 = np.zeros((V, V))
    P2 = np.zeros((V, V, V))
    for j, (x0, x1) in enumerate(xs):
        if a0[j] < 1.0:
            P0 += w[j] * (1 - a0[j]) * m_rej0[j]
        if a1[j] < 1.0:
            P1[x0] += w[j] * a0[j] * (1 - a1[j]) * m_rej1[j]
        P2[x0, x1] += w[j] * a0[j] * a1[j] * m_all[j]
    mn0, mn1 = np.minimum(p0, q0), np.minimum(p1, q1)
    assert np.allclose(P0, np.maximum(0, p0 - q0), rtol=0, atol=1e-12)
    assert np.allclose(P1, mn0[:, None] * np.maximum(0, p1 - q1)[None, :], rtol=0, atol=1e-12)
    assert np.allclose(P2, mn0[:, None, None] * mn1[None, :, None] * p2[None, None, :],
                       rtol=0, atol=1e-12)
    assert np.allclose(P0 + P1.sum(1) + P2.sum((1, 2)), p0, rtol=0, atol=1e-12)


def lossless_cases(seed=1):
    """Small rows for the enumeration: random pairs, the temperature-ratio pair
    (q from 0.8 x the target logits, as in the theory page's simulation), and
    rows where some tokens have p > q and others p < q by a wide margin."""
    rng = np.random.default_rng(seed)
    cases = []
    for V in (2, 3, 5, 8):
        t = rng.normal(0, 2, (3, V)).astype(np.float32)
        d = (t[:2] + rng.normal(0, 1, (2, V))).astype(np.float32)
        cases.append(Rows(t, d, 1.0))
    t = rng.normal(0, 2, (3, 6)).astype(np.float32)
    cases.append(Rows(t, (0.8 * t[:2]).astype(np.float32), 1.0))
    t = rng.normal(0, 3, (3, 7)).astype(np.float32)
    d = (t[:2] + rng.normal(0, 2, (2, 7))).astype(np.float32)
    cases.append(Rows(t, d, 0.7))
    return cases


# --------------------------------------------------------------------------
# Expected tokens per step (closed form) by Monte Carlo
# --------------------------------------------------------------------------
def two_token_rows(a, b):
    """V = 2 rows with p = (a, 1-a), q = (b, 1-b) up to float32 logit rounding."""
    t = np.log(np.array([a, 1 - a])).astype(np.float32)
    d = np.log(np.array([b, 1 - b])).astype(np.float32)
    return t, d


def check_expected_tokens(oracle, gamma, a=0.8, b=0.5, trials=400_000, seed=7):
    """Mean of num_accepted + 1 matches (1 - alpha^(gamma+1)) / (1 - alpha).

    alpha = sum_v min(p, q) is computed with scipy from the float32 logits.
    (disassemble-channel 'Speculative Decoding', section 'Expected number of
    accepted tokens'.)  Same rows at every position, drafts drawn from q.
    """
    t, d = two_token_rows(a, b)
    p = scipy_softmax(t.astype(np.float64))
    q = scipy_softmax(d.astype(np.float64))
    alpha = float(np.minimum(p, q).sum())
    rng = np.random.Generator(np.random.Philox(seed))
    G = gamma
    tgt = np.broadcast_to(t, (trials, G + 1, 2)).copy()
    dft = np.broadcast_to(d, (trials, G, 2)).copy()
    tokens = (rng.random((trials, G)) >= q[0]).astype(np.int32)  # token 0 w.p. q[0]
    u = rng.random((trials, G + 1), dtype=np.float32)
    r = oracle.sample(tgt, dft, tokens, np.full(trials, G, np.int32), u,
                      np.ones(trials, np.float32))
    n = r["num_accepted"] + 1
    expect = (1 - alpha ** (G + 1)) / (1 - alpha)
    se = n.std() / math.sqrt(trials)
    assert abs(n.mean() - expect) < 5 * se, (n.mean(), expect, se)
    # the emitted count follows the truncated geometric law, not just its mean
    for k in range(G):
        pk = alpha ** k * (1 - alpha)
        frac = np.mean(r["num_accepted"] == k)
        assert abs(frac - pk) < 5 * math.sqrt(pk * (1 - pk) / trials) + 1e-12, (k, frac, pk)
    return alpha, n.mean(), expect


# --------------------------------------------------------------------------
# Exact special cases
# --------------------------------------------------------------------------
def check_q_equals_p_accepts_all(oracle, seed=3):
    """Draft rows are bitwise copies of the target rows: ratio is exactly 1, so
    every draft is accepted for any u < 1 and gamma + 1 tokens come out
    (alpha = 1 case of the closed form)."""
    rng = np.random.default_rng(seed)
    B, G, V = 64, 4, 50
    t = rng.normal(0, 3, (B, G + 1, V)).astype(np.float32)
    d = t[:, :G].copy()
    tokens = rng.integers(0, V, (B, G)).astype(np.int32)
    u = rng.random((B, G + 1))
    u[:, :G] = np.maximum(u[:, :G], ONE_MINUS * (rng.random((B, G)) < 0.3))
    r = oracle.sample(t, d, tokens, np.full(B, G, np.int32), u,
                      rng.uniform(0.3, 2.0, B).astype(np.float32))
    assert np.all(r["num_accepted"] == G)
    assert np.array_equal(r["out_tokens"][:, :G], tokens)
    assert np.all((r["out_tokens"][:, G] >= 0) & (r["out_tokens"][:, G] < V))


def check_disjoint_rejects_all(oracle, seed=4):
    """Disjoint supports (alpha = 0): every draft has p(x) = 0, so position 0 is
    always rejected and exactly one token, drawn from p, comes out (E[N] = 1)."""
    rng = np.random.default_rng(seed)
    B, G, V = 200, 3, 8
    t = np.full((B, G + 1, V), -1.0e4, np.float32)
    d = np.full((B, G, V), -1.0e4, np.float32)
    t[:, :, :4] = rng.normal(0, 1, (B, G + 1, 4))
    d[:, :, 4:] = rng.normal(0, 1, (B, G, 4))
    tokens = rng.integers(4, 8, (B, G)).astype(np.int32)
    r = oracle.sample(t, d, tokens, np.full(B, G, np.int32), rng.random((B, G + 1)),
                      np.ones(B, np.float32))
    assert np.all(r["num_accepted"] == 0)
    assert np.all(r["out_tokens"][:, 0] < 4)
    assert np.all(r["out_tokens"][:, 1:] == -1)


def check_greedy_same_rows(oracle, seed=5):
    """Greedy with p == q: drafts are the target argmax, so all are accepted and
    the bonus is the argmax of row gamma_b."""
    rng = np.random.default_rng(seed)
    B, G, V = 40, 5, 300
    t = rng.normal(0, 3, (B, G + 1, V)).astype(np.float32)
    am = t.argmax(axis=2).astype(np.int32)
    gamma = rng.integers(0, G + 1, B).astype(np.int32)
    tokens = am[:, :G].copy()
    for b in range(B):
        tokens[b, gamma[b]:] = 0
    r = oracle.greedy(t, tokens, gamma)
    assert np.array_equal(r["num_accepted"], gamma)
    for b in range(B):
        g = gamma[b]
        assert np.array_equal(r["out_tokens"][b, :g + 1], am[b, :g + 1])
        assert np.all(r["out_tokens"][b, g + 1:] == -1)


def check_greedy_worked_example(oracle):
    """The K = 3 worked example of the 'draft length by load' page (golden file)."""
    ex = json.load(open(os.path.join(GOLDEN, "greedy_worked_example.json")))
    vocab = {w: i for i, w in enumerate(ex["vocab"])}
    V = len(vocab)
    t = np.zeros((1, 4, V), np.float32)
    for i, w in enumerate(ex["target_argmax"]):
        t[0, i, :] = np.linspace(-1, 1, V)[::-1] * 0.1  # small distractors
        t[0, i, vocab[w]] = 5.0
    for draft, out, nacc in ((ex["draft"], ex["expected_out"], ex["expected_num_accepted"]),
                             (ex["all_right_draft"], ex["all_right_expected_out"],
                              ex["all_right_expected_num_accepted"])):
        tok = np.array([[vocab[w] for w in draft]], np.int32)
        r = oracle.greedy(t, tok, np.array([3], np.int32))
        got = [ex["vocab"][i] for i in r["out_tokens"][0] if i >= 0]
        assert got == out and r["num_accepted"][0] == nacc, (got, out)


def check_greedy_ties(oracle):
    """Argmax ties resolve to the lowest token id."""
    t = np.zeros((1, 2, 6), np.float32)
    t[0, 0, [2, 4]] = 3.0
    t[0, 1, [1, 5]] = 7.0
    r = oracle.greedy(t, np.array([[2]], np.int32), np.array([1], np.int32))
    assert r["num_accepted"][0] == 1 and list(r["out_tokens"][0]) == [2, 1]
    r = oracle.greedy(t, np.array([[4]], np.int32), np.array([1], np.int32))
    assert r["num_accepted"][0] == 0 and list(r["out_tokens"][0]) == [2, -1]
    assert r["exact_tie"][0, 0] == 1


def check_inverse_cdf_boundaries(oracle):
    """Bonus draw over four equal logits: p = 1/4 each, so the inclusive
    prefix is exactly 0.25, 0.5, 0.75, 1.0 and token j is chosen for
    u in [j/4, (j+1)/4): the smallest j with C_j > u*S."""
    cases = [(0.0, 0), (0.2499, 0), (0.25, 1), (0.4999999, 1), (0.5, 2), (0.75, 3),
             (float(ONE_MINUS), 3)]
    n = len(cases)
    t = np.zeros((n, 1, 4), np.float32)
    u = np.array([[c[0]] for c in cases])
    r = oracle.sample(t, np.zeros((n, 0, 4), np.float32), np.zeros((n, 0), np.int32),
                      np.zeros(n, np.int32), u, np.ones(n, np.float32))
    assert list(r["out_tokens"][:, 0]) == [c[1] for c in cases]
    assert np.all(r["num_accepted"] == 0)


def check_gamma0_bonus_only(oracle, seed=6):
    """gamma_b = 0 emits one token drawn from p_0 by the final uniform: for
    unequal p the boundaries sit at the cumulative sums of p (scipy)."""
    rng = np.random.default_rng(seed)
    V = 5
    t = rng.normal(0, 1, (1, 1, V)).astype(np.float32)
    p = scipy_softmax(t[0, 0].astype(np.float64))
    c = np.cumsum(p)
    u = np.concatenate([c[:-1] - 1e-9, c[:-1] + 1e-9])
    n = len(u)
    r = oracle.sample(np.repeat(t, n, 0), np.zeros((n, 0, V), np.float32),
                      np.zeros((n, 0), np.int32), np.zeros(n, np.int32), u.reshape(n, 1),
                      np.ones(n, np.float32))
    expect = np.concatenate([np.arange(V - 1), np.arange(1, V)])
    assert np.array_equal(r["out_tokens"][:, 0], expect)


def check_masked_tokens(oracle):
    """-inf logits carry zero probability and are never emitted; a draft token
    with q(x) = 0 is accepted (the ratio's denominator vanishes)."""
    V = 6
    t = np.array([[[0.0, -np.inf, 1.0, -np.inf, 0.5, 0.0],
                   [-np.inf, 2.0, 0.0, 0.0, -np.inf, 1.0]]], np.float32)
    d = np.array([[[1.0, 0.0, -np.inf, 0.0, 0.0, 0.0]]], np.float32)
    n = 200
    rng = np.random.default_rng(8)
    u = rng.random((n, 2))
    u[:, 0] = ONE_MINUS  # force rejection whenever ratio < 1
    tokens = np.ones((n, 1), np.int32)  # p(1) = 0 at position 0: always rejected
    r = oracle.sample(np.repeat(t, n, 0), np.repeat(d, n, 0), tokens, np.ones(n, np.int32),
                      u, np.ones(n, np.float32))
    assert np.all(r["num_accepted"] == 0)
    assert not np.any(np.isin(r["out_tokens"][:, 0], [1, 3]))
    tokens2 = np.full((n, 1), 2, np.int32)  # q(2) = 0: accepted, then bonus from row 1
    r = oracle.sample(np.repeat(t, n, 0), np.repeat(d, n, 0), tokens2, np.ones(n, np.int32),
                      u, np.ones(n, np.float32))
    assert np.all(r["num_accepted"] == 1)
    assert not np.any(np.isin(r["out_tokens"][:, 1], [0, 4]))


def check_softmax(oracle, seed=9):
    """Softmax against closed forms and scipy: uniform logits give 1/V; two
    logits give the logistic function of their difference over T; random rows
    (float32 and bf16) match scipy to 1e-14 relative; huge logits do not
    overflow; the result sums to 1."""
    rng = np.random.default_rng(seed)
    for V in (1, 3, 1000):
        p = oracle.softmax_row(np.full(V, 2.5, np.float32), 0.7)
        assert np.allclose(p, 1.0 / V, rtol=1e-15, atol=0)
    for a, b, T in ((0.0, 1.0, 1.0), (3.0, -2.0, 0.5), (1.5, 1.25, 2.0)):
        p = oracle.softmax_row(np.array([a, b], np.float32), T)
        expect0 = 1.0 / (1.0 + math.exp((np.float64(np.float32(b)) - np.float64(np.float32(a)))
                                        / np.float64(np.float32(T))))
        assert abs(p[0] - expect0) < 1e-15 and abs(p.sum() - 1) < 1e-15
    for T in (0.5, 1.0, 1.7):
        T = float(np.float32(T))
        z = rng.normal(0, 3, 4097).astype(np.float32)
        p = oracle.softmax_row(z, T)
        # (z - m)/T and z/T - max(z/T) round differently: ~eps * |argument|
        ref = scipy_softmax(z.astype(np.float64) / T)
        assert np.allclose(p, ref, rtol=1e-13, atol=0)
        assert abs(p.sum() - 1.0) < 1e-14
        zb = (z.view(np.uint32) >> 16).astype(np.uint16)           # bf16 by truncation
        widened = (zb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        pb = oracle.softmax_row(zb, T)
        assert np.allclose(pb, scipy_softmax(widened / T), rtol=1e-13, atol=0)
    big = np.array([1.0e4, 1.0e4 - 1.0, -1.0e4], np.float32)
    p = oracle.softmax_row(big, 1.0)
    assert np.all(np.isfinite(p)) and abs(p[0] - 1 / (1 + math.exp(-1))) < 1e-15


def check_p_q_at_tokens(oracle, seed=10):
    """The reported p(x_i), q(x_i) equal scipy's softmax at the draft tokens."""
    rng = np.random.default_rng(seed)
    B, G, V = 6, 3, 257
    t = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    d = (t[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    tokens = rng.integers(0, V, (B, G)).astype(np.int32)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    u = np.zeros((B, G + 1))  # accept everything with ratio > 0
    r = oracle.sample(t, d, tokens, np.full(B, G, np.int32), u, T)
    for b in range(B):
        for i in range(G):
            pt = scipy_softmax(t[b, i].astype(np.float64) / np.float64(T[b]))[tokens[b, i]]
            qt = scipy_softmax(d[b, i].astype(np.float64) / np.float64(T[b]))[tokens[b, i]]
            assert abs(r["p_tok"][b, i] / pt - 1) < 1e-13
            assert abs(r["q_tok"][b, i] / qt - 1) < 1e-13


def check_truncation_and_padding(oracle, seed=11):
    """out_tokens holds x_0..x_{k-1} then one drawn token, then -1; uniforms
    that all accept give gamma_b + 1 tokens; ragged gamma_b respected."""
    rng = np.random.default_rng(seed)
    B, G, V = 30, 4, 20
    t = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    d = (t[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    tokens = rng.integers(0, V, (B, G)).astype(np.int32)
    gamma = rng.integers(0, G + 1, B).astype(np.int32)
    u = rng.random((B, G + 1))
    r = oracle.sample(t, d, tokens, gamma, u, np.ones(B, np.float32))
    for b in range(B):
        k = r["num_accepted"][b]
        assert 0 <= k <= gamma[b]
        assert np.array_equal(r["out_tokens"][b, :k], tokens[b, :k])
        assert 0 <= r["out_tokens"][b, k] < V
        assert np.all(r["out_tokens"][b, k + 1:] == -1)
        if k < gamma[b]:
            assert not (u[b, k] < r["p_tok"][b, k] / r["q_tok"][b, k])
        for i in range(k):
            assert u[b, i] < r["p_tok"][b, i] / r["q_tok"][b, i]


def check_accept_strict(oracle):
    """Acceptance is strict: u < p(x)/q(x).  Equal logits make the probabilities
    exact: p uniform over 4 tokens (1/4), q uniform over the first 2 (1/2), so
    the ratio at token 0 is exactly 0.5; u = 0.5 rejects, the double just below
    accepts."""
    t = np.zeros((2, 2, 4), np.float32)
    d = np.array([[[0.0, 0.0, -np.inf, -np.inf]]] * 2, np.float32)
    u = np.array([[0.5, 0.3], [np.nextafter(0.5, 0.0), 0.3]])
    r = oracle.sample(t, d, np.zeros((2, 1), np.int32), np.ones(2, np.int32), u,
                      np.ones(2, np.float32))
    assert list(r["num_accepted"]) == [0, 1], r["num_accepted"]
    assert r["p_tok"][0, 0] == 0.25 and r["q_tok"][0, 0] == 0.5


def check_vanished_residual_falls_back_to_p(oracle):
    """The residual's fallback ([theory], modified-distribution code: draw from
    p when sum max(0, p - q) is zero), on a case fixed by hand.  V = 2, T = 1,
    target row (0, 50), draft row (0, 49.75), draft token 0: in float64
    1 + e^-50 == 1 and 1 + e^-49.75 == 1, so p = (e^-50, 1) and
    q = (e^-49.75, 1) with no rounding in the sums; the ratio e^-0.25 ~ 0.78
    rejects at u = 0.9 and max(0, p - q) is (0, 0).  The draw then follows p's
    inverse CDF: u = 0 gives token 0 (p_0 > 0, which an argmax fallback would
    not give), u = 2.2e-22 lies between p_0 = e^-50 ~ 1.93e-22 and
    q_0 = e^-49.75 ~ 2.48e-22 and gives token 1 (a fallback to q would give
    0).  The reported residual mass is exactly 0."""
    assert 1.0 + math.exp(-50.0) == 1.0 and 1.0 + math.exp(-49.75) == 1.0
    assert math.exp(-50.0) < 2.2e-22 < math.exp(-49.75)
    n = 2
    t = np.array([[[0.0, 50.0], [0.0, 0.0]]] * n, np.float32)
    d = np.array([[[0.0, 49.75]]] * n, np.float32)
    u = np.array([[0.9, 0.0], [0.9, 2.2e-22]])
    r = oracle.sample(t, d, np.zeros((n, 1), np.int32), np.ones(n, np.int32), u,
                      np.ones(n, np.float32))
    assert list(r["num_accepted"]) == [0, 0], r["num_accepted"]
    assert list(r["out_tokens"][:, 0]) == [0, 1], r["out_tokens"]
    assert np.all(r["out_tokens"][:, 1] == -1)
    assert np.all(r["resid_mass"] == 0.0), r["resid_mass"]


def check_subnormal_residual_draw(oracle):
    """The inverse CDF's rounding case, fixed by hand: a residual whose whole
    mass is subnormal, where u*S rounds up to S.  V = 5, T = 1, target row
    (0, 2, 1, -1000, 741), draft row (1, 1, 0.5, -1000, 741), draft token 0.
    Both sums are 1 + (subnormals) == 1, so p_v = e^(z_v - 741),
    q_v = e^(y_v - 741): p_0/q_0 ~ e^-1 rejects at u = 0.9 and the residual
    max(0, p - q) is positive at tokens 1 and 2 only (r_1 ~ 139, r_2 ~ 34 units
    of 2^-1074, tokens 3 and 4 exactly 0).  u = 0.5 selects token 1
    (r_1 > r_2).  u = 1 - 2^-53 makes u*S round to S, where no prefix exceeds
    u*S; the exact u*S < S selects the last token of positive weight, 2 (not
    0, not V - 1, not the largest weight 1).  The reported mass is that
    subnormal sum."""
    sub = lambda x: 0.0 < x < np.finfo(np.float64).tiny  # noqa: E731
    assert sub(math.exp(-739.0)) and sub(math.exp(-741.0))
    n = 2
    t = np.array([[[0.0, 2.0, 1.0, -1000.0, 741.0], [0.0] * 5]] * n, np.float32)
    d = np.array([[[1.0, 1.0, 0.5, -1000.0, 741.0]]] * n, np.float32)
    u = np.array([[0.9, 0.5], [0.9, float(ONE_MINUS)]])
    r = oracle.sample(t, d, np.zeros((n, 1), np.int32), np.ones(n, np.int32), u,
                      np.ones(n, np.float32))
    assert list(r["num_accepted"]) == [0, 0], r["num_accepted"]
    assert list(r["out_tokens"][:, 0]) == [1, 2], r["out_tokens"]
    assert np.all(sub(m) for m in r["resid_mass"]), r["resid_mass"]

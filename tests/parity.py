"""GPU-vs-oracle comparison with near-tie accounting.

The bar: out_tokens and num_accepted identical to the float64 oracle, except
at decisions whose float64 margin is below 1e-6.  Three kinds of decision
have a margin:
  - an acceptance test: |u - ratio|;
  - a draw: the distance of u*S to the nearer CDF edge over S (in units of
    the uniform, like the acceptance margin);
  - the residual itself after a rejection: its float64 mass S.  Below 1e-6
    the residual max(0, p - q) is cancellation at the level of the GPU's
    float32 rounding of p and q (about 1e-7 of each term), so which tokens
    keep weight, and whether the residual vanishes and the draw falls back to
    p, is decided by rounding.
Those are counted as near ties, per kind; any other difference is a mismatch
and must not occur.  p(x_i), q(x_i) must agree within 1e-5 relative at every
position both sides evaluated.
"""
from __future__ import annotations

from dataclasses import asdict, dataclass, field

import numpy as np

NEAR_TIE = 1e-6
PROB_RTOL = 1e-5


@dataclass
class Report:
    requests: int = 0
    accept_decisions: int = 0
    draws: int = 0
    near_tie_accept: int = 0      # oracle margin < 1e-6 (whether or not the sides differ)
    near_tie_cdf: int = 0
    near_tie_resid: int = 0       # rejections whose residual mass is below 1e-6
    differ_near_tie: int = 0      # differences explained by a near tie
    mismatches: list = field(default_factory=list)
    max_prob_rel_err: float = 0.0

    def summary(self):
        return (f"{self.requests} requests, {self.accept_decisions} acceptance tests, "
                f"{self.draws} draws; near ties: accept {self.near_tie_accept}, "
                f"cdf {self.near_tie_cdf}, residual mass {self.near_tie_resid}; "
                f"differences at near ties {self.differ_near_tie}; "
                f"mismatches {len(self.mismatches)}; max p/q rel err {self.max_prob_rel_err:.2e}")

    def to_dict(self):
        d = asdict(self)
        d["mismatches"] = len(self.mismatches)
        return d


def _prob_err(rep, b, p_g, q_g, ref, upto):
    """p/q relative error at positions [0, upto) that both sides evaluated."""
    for arr_g, arr_r in ((p_g, ref["p_tok"][b]), (q_g, ref["q_tok"][b])):
        arr_g, arr_r = arr_g[:upto], arr_r[:upto]
        ok_r, ok_g = ~np.isnan(arr_r), ~np.isnan(arr_g)
        if not np.array_equal(ok_r, ok_g):
            rep.mismatches.append((b, "p/q evaluated set", ok_r.tolist(), ok_g.tolist(), 0))
            continue
        if ok_r.any():
            rel = np.abs(arr_g[ok_r] / arr_r[ok_r] - 1.0)
            rep.max_prob_rel_err = max(rep.max_prob_rel_err, float(rel.max()))


def compare_sample(ref, out_tokens, num_accepted, gamma, p_tok=None, q_tok=None, rep=None):
    """ref: oracle.sample() dict; the rest numpy arrays from the GPU."""
    rep = rep or Report()
    B = len(gamma)
    mass = ref.get("resid_mass")
    for b in range(B):
        rep.requests += 1
        gb = int(gamma[b])
        kr, kg = int(ref["num_accepted"][b]), int(num_accepted[b])
        ma = ref["margin_accept"][b]
        evaluated = min(kr + 1, gb)
        rep.accept_decisions += evaluated
        rep.near_tie_accept += int(np.sum(ma[:evaluated] < NEAR_TIE))
        rep.draws += 1
        cdf_tie = bool(ref["margin_cdf"][b] < NEAR_TIE)
        resid_tie = bool(kr < gb and mass is not None and mass[b] < NEAR_TIE)
        rep.near_tie_cdf += int(cdf_tie)
        rep.near_tie_resid += int(resid_tie)
        if p_tok is not None:
            # positions both sides evaluated: 0..min(kr, kg) (the first
            # rejection included), whether or not the counts agree
            _prob_err(rep, b, p_tok[b], q_tok[b], ref, min(kr, kg) + 1)
        if kr != kg:
            i = min(kr, kg)
            if ma[i] < NEAR_TIE:
                rep.differ_near_tie += 1
            else:
                rep.mismatches.append((b, "num_accepted", kr, kg, float(ma[i])))
            continue
        if not np.array_equal(ref["out_tokens"][b], out_tokens[b]):
            same_rest = np.array_equal(ref["out_tokens"][b][:kr], out_tokens[b][:kr]) and \
                np.array_equal(ref["out_tokens"][b][kr + 1:], out_tokens[b][kr + 1:])
            if same_rest and (cdf_tie or resid_tie):
                rep.differ_near_tie += 1
            else:
                rep.mismatches.append((b, "out_tokens", ref["out_tokens"][b].tolist(),
                                       out_tokens[b].tolist(), float(ref["margin_cdf"][b])))
    return rep


def compare_greedy(ref, out_tokens, num_accepted):
    """Greedy must be bit-exact (ties resolve to the lowest id on both sides)."""
    bad = []
    for b in range(len(num_accepted)):
        if int(ref["num_accepted"][b]) != int(num_accepted[b]) or \
                not np.array_equal(ref["out_tokens"][b], out_tokens[b]):
            bad.append((b, ref["out_tokens"][b].tolist(), out_tokens[b].tolist()))
    return bad

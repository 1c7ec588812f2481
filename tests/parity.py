"""GPU-vs-oracle comparison with near-tie accounting.

The bar: out_tokens and num_accepted identical to the float64 oracle, except
at decisions whose float64 margin is below 1e-6 (|u - ratio| for an
acceptance test, the distance of u*S to the nearer CDF edge over S for a
draw).  Those are counted as near ties, per kind; any other difference is a
mismatch and must not occur.  p(x_i), q(x_i) must agree within 1e-5 relative.
"""
from __future__ import annotations

from dataclasses import dataclass, field

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
    differ_near_tie: int = 0      # differences explained by a near tie
    mismatches: list = field(default_factory=list)
    max_prob_rel_err: float = 0.0

    def summary(self):
        return (f"{self.requests} requests, {self.accept_decisions} acceptance tests, "
                f"{self.draws} draws; near ties: accept {self.near_tie_accept}, "
                f"cdf {self.near_tie_cdf}; differences at near ties {self.differ_near_tie}; "
                f"mismatches {len(self.mismatches)}; max p/q rel err {self.max_prob_rel_err:.2e}")


def compare_sample(ref, out_tokens, num_accepted, gamma, p_tok=None, q_tok=None, rep=None):
    """ref: oracle.sample() dict; the rest numpy arrays from the GPU."""
    rep = rep or Report()
    B = len(gamma)
    for b in range(B):
        rep.requests += 1
        kr, kg = int(ref["num_accepted"][b]), int(num_accepted[b])
        ma = ref["margin_accept"][b]
        evaluated = min(kr + 1, int(gamma[b]))
        rep.accept_decisions += evaluated
        rep.near_tie_accept += int(np.sum(ma[:evaluated] < NEAR_TIE))
        rep.draws += 1
        if ref["margin_cdf"][b] < NEAR_TIE:
            rep.near_tie_cdf += 1
        if kr != kg:
            i = min(kr, kg)
            if ma[i] < NEAR_TIE:
                rep.differ_near_tie += 1
            else:
                rep.mismatches.append((b, "num_accepted", kr, kg, float(ma[i])))
            continue
        if not np.array_equal(ref["out_tokens"][b], out_tokens[b]):
            same_prefix = np.array_equal(ref["out_tokens"][b][:kr], out_tokens[b][:kr]) and \
                np.array_equal(ref["out_tokens"][b][kr + 1:], out_tokens[b][kr + 1:])
            if same_prefix and ref["margin_cdf"][b] < NEAR_TIE:
                rep.differ_near_tie += 1
            else:
                rep.mismatches.append((b, "out_tokens", ref["out_tokens"][b].tolist(),
                                       out_tokens[b].tolist(), float(ref["margin_cdf"][b])))
        if p_tok is not None:
            for arr_g, arr_r in ((p_tok[b], ref["p_tok"][b]), (q_tok[b], ref["q_tok"][b])):
                ok_r, ok_g = ~np.isnan(arr_r), ~np.isnan(arr_g)
                if not np.array_equal(ok_r, ok_g):
                    rep.mismatches.append((b, "p/q evaluated set", ok_r.tolist(), ok_g.tolist(), 0))
                    continue
                if ok_r.any():
                    rel = np.abs(arr_g[ok_r] / arr_r[ok_r] - 1.0)
                    rep.max_prob_rel_err = max(rep.max_prob_rel_err, float(rel.max()))
    return rep


def compare_greedy(ref, out_tokens, num_accepted):
    """Greedy must be bit-exact (ties resolve to the lowest id on both sides)."""
    bad = []
    for b in range(len(num_accepted)):
        if int(ref["num_accepted"][b]) != int(num_accepted[b]) or \
                not np.array_equal(ref["out_tokens"][b], out_tokens[b]):
            bad.append((b, ref["out_tokens"][b].tolist(), out_tokens[b].tolist()))
    return bad

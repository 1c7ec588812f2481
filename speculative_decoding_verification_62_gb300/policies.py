"""Host-side draft-length policies that consume the verify step's outputs.

The verify kernel returns num_accepted per request; a serving loop uses it to
choose the next draft length.  This module holds the policies the pages
describe, written as plain host logic (no GPU work):

* ``BatchSizeTable``: a user table mapping ranges of the number of concurrent
  requests to a draft length K, looked up every step ("speculative decoding:
  draft length by load", the section on vLLM's per-batch-size setting; the
  docs' example maps 1-64 requests to K=3, 65-128 to K=1 and 129-512 to K=0).
* ``AcceptLengthEMA``: per batch-size range, an exponential moving average of
  the number of accepted tokens per verify; the next number of draft steps is
  about round(average) + 1, kept between the smallest and largest candidate,
  and fixed at 1 from 32 concurrent requests on (same page, the section on
  SGLang's adaptive setting; default candidates 1, 3, 7).
* ``AcceptanceEstimator`` and ``optimal_gamma``: an online estimate of the
  per-position acceptance rate alpha from (gamma, num_accepted) pairs, and the
  draft length that maximises the expected speedup
  (1 - alpha^(gamma+1)) / ((1 - alpha)(c gamma + 1)) for a draft/target cost
  ratio c (the explainer of "Fast Inference from Transformers via Speculative
  Decoding", speedup bound and optimal draft length; "Speculative Decoding
  theory", speedup estimate).

Readings where the pages leave a step open: the EMA weight is a parameter
(default 0.2), "round" is round-half-to-even as in Python, and a batch size
outside every table range gets K = 0 (no speculation).
"""
from __future__ import annotations

from dataclasses import dataclass, field


# ---------------------------------------------------------------------------
# Expected tokens and speedup (closed forms)
# ---------------------------------------------------------------------------
def expected_tokens(alpha: float, gamma: int) -> float:
    """E[tokens per verify] = (1 - alpha^(gamma+1)) / (1 - alpha); gamma + 1 at alpha = 1."""
    if gamma < 0:
        raise ValueError("gamma must be >= 0")
    if not 0.0 <= alpha <= 1.0:
        raise ValueError("alpha must be in [0, 1]")
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def speedup(alpha: float, gamma: int, c: float) -> float:
    """Expected speedup over plain decoding: E[tokens] / (c gamma + 1)."""
    if c < 0.0:
        raise ValueError("c must be >= 0")
    return expected_tokens(alpha, gamma) / (c * gamma + 1.0)


def optimal_gamma(alpha: float, c: float, gamma_max: int = 16) -> int:
    """The draft length in [0, gamma_max] with the largest expected speedup
    (smallest such gamma on ties)."""
    best, best_g = -1.0, 0
    for g in range(gamma_max + 1):
        s = speedup(alpha, g, c)
        if s > best * (1.0 + 1e-12):
            best, best_g = s, g
    return best_g


# ---------------------------------------------------------------------------
# Online acceptance-rate estimate
# ---------------------------------------------------------------------------
@dataclass
class AcceptanceEstimator:
    """Estimate of the per-position acceptance rate alpha from verify outputs.

    With independent positions accepted with probability alpha, a verify with
    draft length gamma that accepted k drafts saw k successes and, when
    k < gamma, one failure.  The estimate is successes / (successes +
    failures) over exponentially decayed counts (decay = 1 keeps everything).
    """
    decay: float = 1.0
    prior_successes: float = 0.0
    prior_failures: float = 0.0
    successes: float = field(init=False)
    failures: float = field(init=False)

    def __post_init__(self):
        if not 0.0 < self.decay <= 1.0:
            raise ValueError("decay must be in (0, 1]")
        self.successes = self.prior_successes
        self.failures = self.prior_failures

    def update(self, gamma, num_accepted) -> float:
        """Add a batch of (gamma_b, num_accepted_b) observations; returns alpha."""
        gs = list(gamma) if hasattr(gamma, "__iter__") else [gamma]
        ks = list(num_accepted) if hasattr(num_accepted, "__iter__") else [num_accepted]
        if len(gs) == 1 and len(ks) > 1:
            gs = gs * len(ks)
        if len(gs) != len(ks):
            raise ValueError("gamma and num_accepted differ in length")
        s = f = 0.0
        for g, k in zip(gs, ks):
            g, k = int(g), int(k)
            if not 0 <= k <= g:
                raise ValueError(f"num_accepted {k} outside [0, {g}]")
            s += k
            f += 1.0 if k < g else 0.0
        self.successes = self.decay * self.successes + s
        self.failures = self.decay * self.failures + f
        return self.alpha

    @property
    def alpha(self) -> float:
        n = self.successes + self.failures
        return self.successes / n if n > 0 else 0.0


# ---------------------------------------------------------------------------
# Policies
# ---------------------------------------------------------------------------
class BatchSizeTable:
    """Draft length by number of concurrent requests, from a user table of
    inclusive ranges (lo, hi) -> K."""

    def __init__(self, table):
        rows = sorted((int(lo), int(hi), int(k)) for (lo, hi), k in dict(table).items())
        for lo, hi, k in rows:
            if lo > hi or lo < 1 or k < 0:
                raise ValueError(f"bad table row {(lo, hi)} -> {k}")
        for (lo1, hi1, _), (lo2, _, _) in zip(rows, rows[1:]):
            if lo2 <= hi1:
                raise ValueError("table ranges overlap")
        self.rows = rows

    @classmethod
    def docs_example(cls) -> "BatchSizeTable":
        """The example of the vLLM documentation that the page quotes."""
        return cls({(1, 64): 3, (65, 128): 1, (129, 512): 0})

    def __call__(self, batch_size: int) -> int:
        for lo, hi, k in self.rows:
            if lo <= batch_size <= hi:
                return k
        return 0


class AcceptLengthEMA:
    """Per batch-size range, an EMA of accepted tokens per verify; next steps =
    round(EMA) + 1 within [min(candidates), max(candidates)], and 1 from
    `large_batch` concurrent requests on."""

    def __init__(self, candidates=(1, 3, 7), weight: float = 0.2,
                 ranges=((1, 1), (2, 3), (4, 7), (8, 15), (16, 31)), large_batch: int = 32):
        if not candidates or min(candidates) < 0:
            raise ValueError("candidates must be non-negative draft lengths")
        if not 0.0 < weight <= 1.0:
            raise ValueError("weight must be in (0, 1]")
        self.lo, self.hi = min(candidates), max(candidates)
        self.weight = weight
        self.ranges = tuple((int(a), int(b)) for a, b in ranges)
        self.large_batch = int(large_batch)
        self.ema = {}  # range index -> EMA of accepted tokens per verify

    def _range(self, batch_size: int):
        for i, (a, b) in enumerate(self.ranges):
            if a <= batch_size <= b:
                return i
        return None

    def steps(self, batch_size: int) -> int:
        """Draft steps for the next verify at this batch size."""
        if batch_size >= self.large_batch:
            return 1
        i = self._range(batch_size)
        if i is None or i not in self.ema:
            return self.hi
        return min(self.hi, max(self.lo, round(self.ema[i]) + 1))

    def observe(self, batch_size: int, num_accepted) -> float | None:
        """Fold the mean accepted tokens of one verify into its range's EMA."""
        i = self._range(batch_size)
        ks = list(num_accepted) if hasattr(num_accepted, "__iter__") else [num_accepted]
        if i is None or not ks:
            return None
        mean = sum(int(k) for k in ks) / len(ks)
        prev = self.ema.get(i)
        self.ema[i] = mean if prev is None else (1.0 - self.weight) * prev + self.weight * mean
        return self.ema[i]


def acceptance_rate(gamma, num_accepted) -> float:
    """Fraction of drafted tokens accepted in one verify (0 if none drafted)."""
    g = sum(int(x) for x in gamma)
    return sum(int(k) for k in num_accepted) / g if g else 0.0


__all__ = ["expected_tokens", "speedup", "optimal_gamma", "AcceptanceEstimator",
           "BatchSizeTable", "AcceptLengthEMA", "acceptance_rate"]

"""Draft length (gamma) chosen from the accepted-length histogram of past verify rounds.

Host-side policy above the verify step.  The rules it follows:

* hncyxsy.com article, section 2.3: one round costs the draft's gamma steps plus one
  target verification (about one target step) and yields (1 - a^(gamma+1)) / (1 - a)
  tokens at a constant per-position acceptance rate a; the speedup over plain decoding is
  that yield over the round's cost in target steps, (1 + c * gamma) with c the draft's
  cost per token relative to a target step.  Section 5.2: the best gamma depends on a
  and on the speed ratio; adjust it from the acceptance history, smoothly, to avoid
  oscillation.
* qwbw.cn article, the dynamic-speculation-length remedy: watch the acceptance rate and
  reduce gamma when it stays low, down to plain decoding.
* jennyma11 blog, "怎么选,以及怎么算收益": the emitted-tokens closed form, and tune gamma
  from the recorded accepted-length distribution.

Readings where the pages stop short (each stated here and in the design notes):

* a is estimated from the histogram under the constant-rate model: a round with a
  accepted drafts out of gamma shows a accepted positions and, when a < gamma, one
  rejected position; a_hat = accepted / (accepted + rejected), both sums decayed by
  `decay` per update (recent rounds weigh more).
* gamma in [0, gamma_max] maximises (1 - a^(g+1)) / ((1 - a)(1 + c g)); gamma = 0 is plain
  decoding (speedup 1).  Smoothness: gamma moves one step per update towards that
  maximum, and only when the estimated speedup there beats the current one by `margin`.
* at gamma = 0 no drafts are verified, so nothing is learned: after `probe_every` updates
  at 0 the controller tries gamma = 1 once.
"""
from __future__ import annotations

from typing import Iterable, Optional


def expected_emitted(alpha: float, gamma: int) -> float:
    """Mean tokens a verify round yields: sum_{k=0..gamma} alpha^k."""
    if gamma <= 0:
        return 1.0
    if alpha >= 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def speedup(alpha: float, gamma: int, draft_cost: float) -> float:
    """Tokens per target-step time of speculative rounds over plain decoding."""
    return expected_emitted(alpha, gamma) / (1.0 + draft_cost * max(gamma, 0))


class GammaController:
    """Tracks the acceptance rate of past rounds and proposes the next round's gamma.

    draft_cost: the draft's cost per token as a fraction of a target step (c above).
    """

    def __init__(self, gamma: int = 4, gamma_max: int = 8, draft_cost: float = 0.1,
                 decay: float = 0.9, margin: float = 0.02, allow_fallback: bool = True,
                 probe_every: int = 32):
        if not (0 <= gamma <= gamma_max) or gamma_max < 1:
            raise ValueError("need 0 <= gamma <= gamma_max and gamma_max >= 1")
        if not (0.0 < decay <= 1.0) or draft_cost < 0.0 or margin < 0.0:
            raise ValueError("need 0 < decay <= 1, draft_cost >= 0, margin >= 0")
        self.gamma = gamma
        self.gamma_max = gamma_max
        self.draft_cost = draft_cost
        self.decay = decay
        self.margin = margin
        self.gamma_min = 0 if allow_fallback else 1
        self.probe_every = probe_every
        self._acc = 0.0   # decayed sum of accepted positions
        self._rej = 0.0   # decayed count of rejected positions
        self._idle = 0    # updates spent at gamma = 0

    @property
    def alpha(self) -> Optional[float]:
        """The estimated per-position acceptance rate (None before any observation)."""
        n = self._acc + self._rej
        return None if n <= 0.0 else self._acc / n

    def observe(self, num_accepted: Iterable[int], gamma_used: int) -> None:
        """Record one round: the accepted draft count of every sequence, out of gamma_used."""
        acc = rej = 0
        for a in num_accepted:
            a = int(a)
            if a < 0 or a > gamma_used:
                raise ValueError(f"accepted count {a} outside [0, {gamma_used}]")
            acc += a
            rej += 1 if a < gamma_used else 0
        self._acc = self.decay * self._acc + acc
        self._rej = self.decay * self._rej + rej

    def best(self) -> Optional[int]:
        """The gamma of largest estimated speedup (ties: the smaller gamma)."""
        a = self.alpha
        if a is None:
            return None
        return max(range(self.gamma_min, self.gamma_max + 1),
                   key=lambda g: (speedup(a, g, self.draft_cost), -g))

    def update(self, num_accepted: Iterable[int], gamma_used: int) -> int:
        """Record one round and return the gamma for the next."""
        if gamma_used > 0:
            self.observe(num_accepted, gamma_used)
        if self.gamma == 0:
            self._idle += 1
            if self._idle >= self.probe_every:
                self._idle = 0
                self.gamma = 1
            return self.gamma
        self._idle = 0
        target = self.best()
        if target is not None and target != self.gamma:
            a = self.alpha
            if speedup(a, target, self.draft_cost) > (1.0 + self.margin) * speedup(
                    a, self.gamma, self.draft_cost):
                self.gamma += 1 if target > self.gamma else -1
        return self.gamma

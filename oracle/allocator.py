"""RateQuant per-component bit allocation.

Source: RateQuant technical summary, Methodology section 1 (problem
formulation and optimal allocation) and section 3 (integer allocation and
extensions):

* Each quantizer's mean-squared error follows D(b) = alpha * beta^-b.
* Objective: minimise sum_i w_i D_i(b_i) subject to sum_i b_i = B, with w_i
  the sensitivity of component i.
* Lagrangian stationarity gives the continuous optimum (reverse
  waterfilling)  b*_i = b_bar + (ln w_i - ln w_bar) / ln beta  with b_bar the
  mean bit-width and w_bar the geometric mean of the sensitivities; the
  achievable reduction of the weighted distortion over uniform allocation is
  bounded by the ratio of the arithmetic to the geometric mean of w.
* The integer allocation is a greedy marginal-gain loop: repeatedly give bits
  to the component whose upgrade lowers the weighted distortion the most,
  until the budget is exhausted.
* K/V decoupling: K and V of every (layer, head) are independent components
  with their own curve (own beta), i.e. 2N components.

Readings:
* alpha is folded into w (w_i here is sensitivity x alpha_i).
* Each component has a set of allowed bit-widths; it starts at its smallest
  allowed width.  A step moves one component to its next allowed width; its
  merit is the gain per bit, w_i (beta_i^-b - beta_i^-b') / (b' - b), the
  plain knapsack reading (equal to the raw gain for unit steps).  Only steps
  that fit in the remaining budget are candidates; ties go to the lowest
  index; the loop stops when no step fits.
* Component order for a cache is ((layer * Hkv + head) * 2 + kv), kv = 0
  for K.
"""
from __future__ import annotations

import itertools
import math
from typing import Sequence


class BudgetError(ValueError):
    """The budget is below the sum of the smallest allowed widths."""


def _next_allowed(allowed: Sequence[int], b: int):
    for x in sorted(allowed):
        if x > b:
            return x
    return None


def greedy(w: Sequence[float], beta: Sequence[float], budget: int,
           allowed: Sequence[Sequence[int]]) -> tuple[list[int], int]:
    """Greedy marginal-gain integer allocation.  Returns (bits, leftover)."""
    n = len(w)
    bits = [min(a) for a in allowed]
    used = sum(bits)
    if used > budget:
        raise BudgetError(f"budget {budget} < minimum allocation {used}")
    while True:
        best, best_gain = -1, 0.0
        for i in range(n):
            nxt = _next_allowed(allowed[i], bits[i])
            if nxt is None:
                continue
            cost = nxt - bits[i]
            if cost > budget - used:
                continue
            gain = float(w[i]) * (float(beta[i]) ** (-bits[i]) - float(beta[i]) ** (-nxt)) / cost
            if best < 0 or gain > best_gain:
                best, best_gain = i, gain
        if best < 0:
            break
        nxt = _next_allowed(allowed[best], bits[best])
        used += nxt - bits[best]
        bits[best] = nxt
    return bits, budget - used


def weighted_distortion(w: Sequence[float], beta: Sequence[float],
                        bits: Sequence[float]) -> float:
    return float(sum(float(wi) * float(be) ** (-float(b)) for wi, be, b in zip(w, beta, bits)))


def closed_form(w: Sequence[float], beta: float, b_bar: float) -> list[float]:
    """Continuous optimum b*_i = b_bar + (ln w_i - ln w_geo) / ln beta (one beta)."""
    logs = [math.log(float(x)) for x in w]
    log_gm = sum(logs) / len(logs)
    return [b_bar + (li - log_gm) / math.log(beta) for li in logs]


def am_gm_ratio(w: Sequence[float]) -> float:
    """Arithmetic mean / geometric mean of the sensitivities."""
    am = sum(float(x) for x in w) / len(w)
    gm = math.exp(sum(math.log(float(x)) for x in w) / len(w))
    return am / gm


def brute_force(w: Sequence[float], beta: Sequence[float], budget: int,
                allowed: Sequence[Sequence[int]]) -> tuple[list[int], float]:
    """Exhaustive minimum of the weighted distortion over all allocations with
    sum(bits) <= budget (tiny n only)."""
    best, best_d = None, math.inf
    for combo in itertools.product(*[sorted(a) for a in allowed]):
        if sum(combo) > budget:
            continue
        dist = weighted_distortion(w, beta, combo)
        if dist < best_d:
            best, best_d = list(combo), dist
    return best, best_d

"""Pins for oracle.allocator (RateQuant greedy, closed form, AM/GM, brute force)."""
import math

import numpy as np
import pytest

from oracle import allocator
from tests.conftest import golden_rows
from workloads import sensitivities


def _golden():
    return {r[0]: r[1:] for r in golden_rows("alloc_closed_form.txt")}


def test_closed_form_hand_example():
    g = _golden()
    w = [float(x) for x in g["w"][0].split()]
    got = allocator.closed_form(w, float(g["beta"][0]), float(g["b_bar"][0]))
    want = [float(x) for x in g["b_star"][0].split()]
    assert np.allclose(got, want, atol=1e-12)
    assert abs(allocator.am_gm_ratio(w) - float(g["am_gm"][0])) < 1e-12
    pair = [float(x) for x in g["am_gm_pair"][0].split()]
    assert abs(allocator.am_gm_ratio(pair) - float(g["am_gm_pair"][1])) < 1e-12


def test_am_gm_is_the_distortion_ratio_at_the_optimum():
    # sum w beta^-b* = n GM(w) beta^-b_bar, while uniform gives n AM(w) beta^-b_bar.
    rng = np.random.default_rng(1)
    w = rng.lognormal(0, 1, 12)
    beta, b_bar = 4.3, 3.0
    bstar = allocator.closed_form(w, beta, b_bar)
    assert abs(sum(bstar) - 12 * b_bar) < 1e-9
    d_opt = allocator.weighted_distortion(w, [beta] * 12, bstar)
    d_uni = allocator.weighted_distortion(w, [beta] * 12, [b_bar] * 12)
    assert abs(d_uni / d_opt - allocator.am_gm_ratio(w)) < 1e-9


@pytest.mark.parametrize("seed", range(12))
def test_greedy_is_optimal_for_unit_steps(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 6))
    w = rng.lognormal(0, 1.5, n)
    beta = rng.uniform(3.0, 6.0, n)
    allowed = [list(range(1, 7))] * n
    budget = int(rng.integers(n, 6 * n + 1))
    bits, left = allocator.greedy(w, beta, budget, allowed)
    _, best = allocator.brute_force(w, beta, budget, allowed)
    assert allocator.weighted_distortion(w, beta, bits) <= best * (1 + 1e-12)
    if budget <= 6 * n:
        assert sum(bits) == budget and left == 0


@pytest.mark.parametrize("seed", range(6))
def test_greedy_nonunit_steps_respects_budget(seed):
    rng = np.random.default_rng(100 + seed)
    n = 6
    w = rng.lognormal(0, 1, n)
    beta = rng.uniform(3.5, 5.5, n)
    allowed = [[4, 8], [2, 4]] * 3
    budget = int(rng.integers(18, 48))
    bits, left = allocator.greedy(w, beta, budget, allowed)
    assert sum(bits) + left == budget and left >= 0
    assert all(b in a for b, a in zip(bits, allowed))
    _, best = allocator.brute_force(w, beta, budget, allowed)
    assert allocator.weighted_distortion(w, beta, bits) >= best * (1 - 1e-12)


def test_greedy_tracks_closed_form():
    rng = np.random.default_rng(7)
    w = rng.lognormal(0, 0.7, 16)
    beta, b_bar = 4.0, 4.0
    bits, _ = allocator.greedy(w, [beta] * 16, int(16 * b_bar), [list(range(0, 13))] * 16)
    bstar = allocator.closed_form(w, beta, b_bar)
    assert sum(bits) == 64
    assert max(abs(b - s) for b, s in zip(bits, bstar)) < 1.0


def test_uniform_weights_give_uniform_bits():
    bits, _ = allocator.greedy([1.0] * 8, [4.0] * 8, 8 * 3 + 3, [list(range(1, 9))] * 8)
    assert sorted(bits) == [3] * 5 + [4] * 3
    assert bits[:3] == [4, 4, 4]                       # ties go to the lowest index


def test_keys_with_larger_weight_get_more_bits():
    # "Quantize What Counts": keys carry more weight than values -> more bits.
    w = [5.0, 1.0] * 4
    bits, _ = allocator.greedy(w, [4.0] * 8, 24, [[2, 4, 8]] * 8)
    for i in range(0, 8, 2):
        assert bits[i] >= bits[i + 1]


def test_budget_error():
    with pytest.raises(allocator.BudgetError):
        allocator.greedy([1.0, 1.0], [4.0, 4.0], 5, [[4, 8], [2, 4]])


def test_mixed_config_average_3_is_the_minimum_allocation():
    # 32 layers x 8 KV heads, K in {4,8}, V in {2,4}: avg 3 bits = the K4V2 floor.
    w = sensitivities(1003, 32, 8).reshape(-1)
    allowed = [[4, 8], [2, 4]] * 256
    beta = [4.0] * 512
    bits, left = allocator.greedy(w, beta, 3 * 512, allowed)
    assert bits == [4, 2] * 256 and left == 0
    bits, left = allocator.greedy(w, beta, int(3.5 * 512), allowed)
    # V steps 2->4 gain far more per bit than K steps 4->8 at equal weights,
    # so the extra 256 bits upgrade V of the most sensitive heads first.
    assert sum(bits) + left == 1792
    assert bits[0::2] == [4] * 256 and sorted(set(bits[1::2])) == [2, 4]
    assert sum(1 for b in bits[1::2] if b == 4) == 128

"""Pins for oracle.fp16 directed rounding against brute force over all fp16 values."""
import numpy as np

from oracle import fp16

ALL = fp16.all_finite_fp16()


def _brute_down(x):
    i = np.searchsorted(ALL, x, side="right") - 1
    return ALL[i]


def _brute_up(x):
    i = np.searchsorted(ALL, x, side="left")
    return ALL[i]


def test_directed_rounding_matches_enumeration():
    rng = np.random.default_rng(5)
    xs = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-7, 5, 20000),
        ALL[1:-1],                                  # exact fp16 values
        np.nextafter(ALL[1:-1], np.inf),            # just above
        np.nextafter(ALL[1:-1], -np.inf),           # just below
        np.array([0.0, 1e-9, -1e-9, 65504.0, -65504.0]),
    ])
    d = fp16.round_down(xs).astype(np.float64)
    u = fp16.round_up(xs).astype(np.float64)
    assert np.array_equal(d, _brute_down(xs))
    assert np.array_equal(u, _brute_up(xs))
    assert np.all(d <= xs) and np.all(u >= xs)


def test_float32_inputs():
    x = np.float32([0.1, 1.6, -0.1, 3.3333333])
    assert np.all(fp16.round_down(x).astype(np.float64) <= x.astype(np.float64))
    assert np.all(fp16.round_up(x).astype(np.float64) >= x.astype(np.float64))

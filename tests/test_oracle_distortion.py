"""Pins for oracle.distortion: exact-curve recovery and the beta range."""
import numpy as np

from oracle import distortion
from workloads import kv_tokens


def test_fit_recovers_an_exact_curve():
    b = np.arange(2, 7)
    alpha, beta = distortion.fit(b, 0.7 * 4.6 ** (-b))
    assert abs(alpha - 0.7) < 1e-10 and abs(beta - 4.6) < 1e-10


def test_fitted_beta_is_in_the_reported_range():
    # RateQuant, Problem statement: beta between about 3.6 and 5.3 for real quantizers.
    x = kv_tokens(4, 0, 1, 2048, 1, 128, 4, 10.0, 50.0)[0, :, 0]
    mse = distortion.measure_mse(x, 128)
    assert np.all(np.diff(mse) < 0)
    _, beta = distortion.fit(range(2, 7), mse)
    assert 3.0 < beta < 6.0

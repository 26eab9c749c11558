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


def test_mse_of_uniform_values_is_step_squared_over_12():
    # Rotated values u_j i.i.d. uniform: the error of a uniform quantizer with
    # step s is uniform on [-s/2, s/2], mean square s^2 / 12 (in u's units);
    # the orthonormal rotation divides it by the block size.  The per-vector
    # step is s = fp16-up((max - fp16-down(min)) / (2^b - 1)).
    from oracle import fp16
    from oracle.hadamard import unrotate
    rng = np.random.default_rng(11)
    block, d, n = 64, 128, 4000
    u = rng.uniform(-3.0, 5.0, size=(n, d))
    x = unrotate(u, block)                     # rotate(x) gives back u
    widths = [4, 5, 6]
    mse = distortion.measure_mse(x, block, widths)
    u32 = u.astype(np.float32)
    z = fp16.round_down(u32.min(axis=1)).astype(np.float64)
    for b, got in zip(widths, mse):
        s = fp16.round_up(((u32.max(axis=1) - z.astype(np.float32)) / np.float32(2 ** b - 1))
                          .astype(np.float32)).astype(np.float64)
        want = np.mean(s ** 2) / 12.0 / block
        assert abs(got / want - 1.0) < 0.03, (b, got, want)


def test_mse_never_exceeds_half_a_step():
    # |u - deq| <= s / 2 for every element (directed rounding of s and z)
    from oracle.hadamard import unrotate
    rng = np.random.default_rng(12)
    u = rng.standard_normal((500, 64)) * rng.uniform(0.1, 30.0, size=(500, 1))
    x = unrotate(u, 32)
    for b in range(1, 9):
        mse = distortion.measure_mse(x, 32, [b])[0]
        span = u.max(axis=1) - u.min(axis=1)
        bound = np.mean((span * 1.01 / (2 ** b - 1)) ** 2) / 4.0 / 32
        assert mse <= bound


def test_mse_is_zero_on_the_grid_of_its_width():
    # u on the 2-bit grid {z, z + s, z + 2s, z + 3s} with fp16-exact z and s and
    # both ends present: the quantizer reproduces it exactly at b = 2 (levels
    # 2^b - 1 = 3), not at b = 3.
    from oracle.hadamard import unrotate
    rng = np.random.default_rng(13)
    z, s = -1.5, 0.75
    c = rng.integers(0, 4, size=(64, 32))
    c[:, 0], c[:, 1] = 0, 3
    x = unrotate(z + s * c, 32)
    mse = distortion.measure_mse(x, 32, [2, 3])
    assert mse[0] == 0.0 and mse[1] > 0.0

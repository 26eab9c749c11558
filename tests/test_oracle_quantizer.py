"""Pins for oracle.quantizer: hand-worked examples, bounds, ties, exact grids."""
import numpy as np
import pytest

from oracle import hadamard, quantizer
from tests.conftest import golden_rows
from workloads import kv_tokens


@pytest.mark.parametrize("row", golden_rows("quant_worked_examples.txt"))
def test_worked_examples(row):
    bits = int(row[0])
    u = np.array(row[1].split(), dtype=np.float32)[None]
    c, s, z = quantizer.quantize(u, bits)
    assert float(s[0]) == float(row[2])
    assert float(z[0]) == float(row[3])
    assert c[0].tolist() == [int(t) for t in row[4].split()]
    deq = quantizer.dequantize(c, s, z)[0]
    assert np.allclose(deq, np.array(row[5].split(), dtype=np.float64), rtol=0, atol=1e-12)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_error_bound_and_range(bits):
    x = kv_tokens(11, 0, 1, 512, 2, 128, 4, 10.0, 50.0)[0].reshape(-1, 128)
    u = hadamard.rotate(x, 128).astype(np.float32)
    s, z = quantizer.scale_zero(u, bits)
    raw = quantizer.codes_given(u, s, z, bits, clip=False)
    m = (1 << bits) - 1
    assert raw.min() >= 0 and raw.max() <= m            # the clamp never fires
    deq = quantizer.dequantize(raw, s, z)
    sf = s.astype(np.float64)[:, None]
    assert np.all(np.abs(u.astype(np.float64) - deq) <= sf / 2 * (1 + 1e-6))
    # z is the largest fp16 <= min, every value inside [z, z + M s]
    assert np.all(z.astype(np.float64) <= u.min(1))
    assert np.all(z.astype(np.float64) + m * sf[:, 0] >= u.max(1) * (1 - 1e-6))
    # the extreme elements take the extreme codes
    rows = np.arange(u.shape[0])
    assert np.all(raw[rows, u.argmin(1)] == 0)
    assert np.all(raw[rows, u.argmax(1)] == m)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_ties_round_to_even(bits):
    m = (1 << bits) - 1
    s = 0.25                                   # dyadic: every tie is exact
    z = -2.0
    ks = np.arange(m)
    u = np.concatenate([[z], z + (ks + 0.5) * s, [z + m * s]]).astype(np.float32)[None]
    c, s16, z16 = quantizer.quantize(u, bits)
    assert float(s16[0]) == s and float(z16[0]) == z
    want = [0] + [k if k % 2 == 0 else k + 1 for k in ks] + [m]
    assert c[0].tolist() == want


def test_8bit_grid_is_lossless():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=(50, 128))
    codes[:, 0], codes[:, 1] = 0, 255
    s, z = 0.03125, -3.5
    u = (z + codes * s).astype(np.float32)
    c, s16, z16 = quantizer.quantize(u, 8)
    assert np.array_equal(c, codes)
    assert np.array_equal(quantizer.dequantize(c, s16, z16), u.astype(np.float64))


def test_rotation_helps_outliers():
    # "SAW-INT4", section 2: rotating before quantizing spreads outlier channels.
    x = kv_tokens(12, 0, 1, 256, 1, 128, 4, 10.0, 50.0)[0, :, 0]
    raw_err = np.mean((quantizer.dequantize(*quantizer.quantize(x, 4)) - x) ** 2)
    u = hadamard.rotate(x, 128).astype(np.float32)
    c, s, z = quantizer.quantize(u, 4)
    rot_err = np.mean((hadamard.unrotate(quantizer.dequantize(c, s, z), 128) - x) ** 2)
    assert rot_err < 0.5 * raw_err


def test_rejects_unsupported_bits():
    with pytest.raises(ValueError):
        quantizer.quantize(np.zeros((1, 4), np.float32), 3)

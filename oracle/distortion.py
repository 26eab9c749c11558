"""Distortion-rate fit D(b) = alpha * beta^-b for this library's quantizer.

Source: RateQuant technical summary, Methodology section 3 (distortion
calibration: fit (alpha, beta) per quantizer instead of assuming one global
beta) and section 4 (pipeline: the fit uses 5 bit-widths); Problem statement
(beta differs between quantizers, e.g. 3.6 to 5.3).

The fit is least squares of ln D(b) = ln alpha - b ln beta over the measured
mean-squared error of quantize/dequantize in the rotated domain, on a sample
of vectors, at b = 2 .. 6.  The quantizer used for the measurement is the one
in ``quantizer`` (this module allows any width 1..8 for the fit only).
"""
from __future__ import annotations

import numpy as np

from . import fp16
from .hadamard import rotate


def _quantize_any(u32: np.ndarray, bits: int) -> np.ndarray:
    """Dequantized float64 values of u32 at any width 1..8 (same rule as
    ``quantizer``, without its restriction to 2/4/8)."""
    m = np.float32((1 << bits) - 1)
    mn = u32.min(axis=-1)
    mx = u32.max(axis=-1)
    z = fp16.round_down(mn)
    span = (mx - z.astype(np.float32)).astype(np.float32)
    s = fp16.round_up((span / m).astype(np.float32))
    sf = s.astype(np.float32)
    zf = z.astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(sf > 0, (np.float32(1.0) / sf).astype(np.float32), np.float32(0))
    diff = (u32 - zf[..., None]).astype(np.float32)
    c = np.rint(diff.astype(np.float64) * inv.astype(np.float64)[..., None])
    c = np.clip(c, 0, float(m))
    return c * sf.astype(np.float64)[..., None] + zf.astype(np.float64)[..., None]


def measure_mse(x: np.ndarray, block: int, widths=(2, 3, 4, 5, 6)) -> np.ndarray:
    """Mean-squared quantization error of rotated vectors x[n, d] per width.

    The error is measured on the orthonormal rotation (u / sqrt(block)) so
    that it is in the units of the original vectors.
    """
    u32 = rotate(x, block).astype(np.float32)
    out = []
    for b in widths:
        deq = _quantize_any(u32, b)
        err = (deq - u32.astype(np.float64)) / np.sqrt(block)
        out.append(float(np.mean(err ** 2)))
    return np.array(out)


def fit(widths, mse) -> tuple[float, float]:
    """Least-squares (alpha, beta) of ln D = ln alpha - b ln beta."""
    b = np.asarray(widths, dtype=np.float64)
    y = np.log(np.asarray(mse, dtype=np.float64))
    a = np.stack([np.ones_like(b), -b], axis=1)
    (ln_alpha, ln_beta), *_ = np.linalg.lstsq(a, y, rcond=None)
    return float(np.exp(ln_alpha)), float(np.exp(ln_beta))

"""Directed rounding of real values to IEEE binary16 (fp16).

The quantizer stores one fp16 scale and one fp16 zero per vector
("SAW-INT4 ...", summary: token-wise INT4; RateQuant technical summary,
Methodology section 3, K/V decoupling: asymmetric per-token quantization).
The zero is rounded toward -inf and the scale toward +inf so that every
value of the vector lies inside [z, z + (2^b - 1) s] for the *stored* values
(a reading of this library; the pages do not say how the pair is rounded).
"""
from __future__ import annotations

import numpy as np

_NEG_INF16 = np.float16(-np.inf)
_POS_INF16 = np.float16(np.inf)


def round_down(x: np.ndarray) -> np.ndarray:
    """Largest fp16 value <= x (elementwise).  x: float32 or float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)          # round to nearest, ties to even
    over = h.astype(np.float64) > x
    with np.errstate(over="ignore"):
        h = np.where(over, np.nextafter(h, _NEG_INF16), h)
    return h.astype(np.float16)


def round_up(x: np.ndarray) -> np.ndarray:
    """Smallest fp16 value >= x (elementwise).  x: float32 or float64."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)
    under = h.astype(np.float64) < x
    with np.errstate(over="ignore"):
        h = np.where(under, np.nextafter(h, _POS_INF16), h)
    return h.astype(np.float16)


def all_finite_fp16() -> np.ndarray:
    """Every finite fp16 value, sorted ascending (float64), -0 dropped."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bits.view(np.float16).astype(np.float64)
    v = v[np.isfinite(v)]
    return np.unique(v)

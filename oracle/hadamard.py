"""Block-diagonal Walsh-Hadamard rotation, by explicit matrix multiply.

Source: "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization for Real-World
LLM Serving", section 2 ("mix before you shrink"): each KV head vector is
rotated by a block-diagonal Hadamard transform before quantization, which
spreads large outlier channels over the block.

Readings (the page names the transform but fixes neither ordering nor
scale):

* Ordering: Sylvester's construction H_1 = [1], H_2n = [[H_n, H_n],
  [H_n, -H_n]], whose entry (i, j) is (-1)^popcount(i & j) (natural order).
* Scale: the cache quantizes the *unnormalised* block transform u = H x
  (entries +-1).  The orthonormal rotation is H / sqrt(n); since H H = n I,
  q . k = (H q) . (H k) / n, and x = H u / n.  Quantization is
  scale-equivariant, so quantizing u instead of (H / sqrt(n)) x yields the
  same codes in exact arithmetic; it only changes the stored fp16 scale and
  zero by the factor sqrt(n).  Using the unnormalised form keeps every
  rescaling a power of two (exact in binary floating point).
"""
from __future__ import annotations

import numpy as np


def sylvester(n: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_n (int64, entries +-1), n a power of two."""
    if n < 1 or n & (n - 1):
        raise ValueError(f"Hadamard order must be a power of two, got {n}")
    h = np.ones((1, 1), dtype=np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def block_hadamard(d: int, n: int) -> np.ndarray:
    """Block-diagonal matrix diag(H_n, ..., H_n) of size d x d (int64)."""
    if d % n:
        raise ValueError(f"block {n} does not divide head_dim {d}")
    out = np.zeros((d, d), dtype=np.int64)
    h = sylvester(n)
    for b in range(d // n):
        out[b * n:(b + 1) * n, b * n:(b + 1) * n] = h
    return out


def rotate(x: np.ndarray, n: int) -> np.ndarray:
    """u = H_blk x along the last axis, in float64 (unnormalised transform)."""
    x = np.asarray(x, dtype=np.float64)
    hb = block_hadamard(x.shape[-1], n).astype(np.float64)
    return x @ hb.T


def unrotate(u: np.ndarray, n: int) -> np.ndarray:
    """x = H_blk u / n along the last axis, in float64 (inverse of ``rotate``)."""
    u = np.asarray(u, dtype=np.float64)
    hb = block_hadamard(u.shape[-1], n).astype(np.float64)
    return (u @ hb.T) / n


def orthonormal(d: int, n: int) -> np.ndarray:
    """The orthonormal block rotation diag(H_n) / sqrt(n), float64."""
    return block_hadamard(d, n).astype(np.float64) / np.sqrt(n)

"""Token-wise asymmetric INT-b quantization with one fp16 scale and zero, and
the per-channel symmetric key quantizer of the key-per-channel mode.

Sources:
* "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization for Real-World LLM
  Serving", summary paragraph: token-wise quantization (one scale per token
  and head) after a block-diagonal Hadamard rotation.
* RateQuant technical summary, Methodology section 3 (K/V decoupling):
  values use asymmetric per-token quantization; keys and values are
  separate components with their own bit-widths.

Definition (per vector u of length d -- one token, one KV head, K or V, after
rotation; M = 2^b - 1):

    mn = min(u), mx = max(u)
    z  = fp16 round-down(mn)
    s  = fp16 round-up( (mx - z) / M )
    c_j = round-half-even( (u_j - z) / s ),  0 <= c_j <= M
    deq_j = c_j * s + z

Readings of steps the pages leave open:
* The scale and zero are floats (not an integer zero point).
* Directed rounding of s and z puts every u_j inside [z, z + M s] for the
  stored fp16 values, hence |u_j - deq_j| <= s / 2.
* The decision that turns a real value into an integer code is taken in
  float32, the precision of the CUDA kernel: u is the exact rotation rounded
  once to float32; mx - z and the division by M are float32 operations with
  round-to-nearest; the code is round-half-even of the exact product
  (u_j - z) * (1 / s) where both the difference and the reciprocal are
  float32-rounded.  This fixes the integers bit for bit given the same u.
* mx == z (a constant vector whose value is fp16-exact) gives s = 0; all codes
  are then 0 and deq = z.
"""
from __future__ import annotations

import numpy as np

from . import fp16


def levels(bits: int) -> int:
    if bits not in (2, 4, 8):
        raise ValueError(f"unsupported bit-width {bits}")
    return (1 << bits) - 1


def scale_zero(u32: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """fp16 (s, z) per vector for float32 vectors u32[..., d]."""
    u32 = np.asarray(u32, dtype=np.float32)
    m = np.float32(levels(bits))
    mn = u32.min(axis=-1)
    mx = u32.max(axis=-1)
    z = fp16.round_down(mn)
    span = (mx - z.astype(np.float32)).astype(np.float32)        # float32 subtract
    s = fp16.round_up((span / m).astype(np.float32))              # float32 divide
    return s, z


def codes_given(u32: np.ndarray, s: np.ndarray, z: np.ndarray, bits: int,
                clip: bool = True) -> np.ndarray:
    """Integer codes of u32[..., d] for given fp16 s[...] and z[...].

    With ``clip=False`` the raw rounded values are returned (as int64) so
    that a test can check that the clamp never fires.
    """
    u32 = np.asarray(u32, dtype=np.float32)
    sf = np.asarray(s, dtype=np.float16).astype(np.float32)
    zf = np.asarray(z, dtype=np.float16).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(sf > 0, (np.float32(1.0) / sf).astype(np.float32), np.float32(0.0))
    diff = (u32 - zf[..., None]).astype(np.float32)               # float32 subtract
    prod = diff.astype(np.float64) * inv.astype(np.float64)[..., None]   # exact product
    c = np.rint(prod).astype(np.int64)                            # half to even
    c = np.where((sf > 0)[..., None], c, 0)
    if clip:
        c = np.clip(c, 0, levels(bits))
    return c


def quantize(u32: np.ndarray, bits: int):
    """(codes uint8[..., d], s fp16[...], z fp16[...]) for float32 vectors."""
    s, z = scale_zero(u32, bits)
    c = codes_given(u32, s, z, bits).astype(np.uint8)
    return c, s, z


def dequantize(codes: np.ndarray, s: np.ndarray, z: np.ndarray) -> np.ndarray:
    """deq = c * s + z in float64."""
    c = np.asarray(codes, dtype=np.float64)
    sf = np.asarray(s, dtype=np.float16).astype(np.float64)
    zf = np.asarray(z, dtype=np.float16).astype(np.float64)
    return c * sf[..., None] + zf[..., None]


def rotate_and_quantize(x: np.ndarray, block: int, bits: int):
    """Rotate bf16 vectors x[..., d] (float32 holding bf16 values) and quantize.

    Returns (codes, s, z, u32) with u32 the float32-rounded exact rotation.
    """
    from .hadamard import rotate
    u32 = rotate(x, block).astype(np.float32)
    c, s, z = quantize(u32, bits)
    return c, s, z, u32


# ------------------------------------------------------------------------
# Per-channel symmetric keys (the key-per-channel mode).
#
# Sources:
# * RateQuant technical summary, Methodology section 3 (K/V decoupling): KIVI
#   quantizes keys symmetrically per channel and values asymmetrically per
#   token, so K and V are separate components.
# * "LogQuant ...", section 5 (implementation): 2-bit quantization with a
#   key-per-channel strategy.
#
# Definition (per group u[n, d] -- the n = 16 tokens of one page of one KV
# head's keys, after rotation; Q = 2^(b-1) - 1):
#
#     s_j = fp16 round-up( max_t |u_tj| / Q )       one scale per channel j
#     c_tj = round-half-even( u_tj / s_j ),  -Q <= c_tj <= Q
#     deq_tj = c_tj * s_j
#
# Readings of steps the pages leave open:
# * The group is one page (16 tokens): the pages give no group size, and the
#   page is the cache's unit of storage.
# * "Symmetric" means no zero point and the level range [-Q, Q] (2^b - 1
#   levels; code -2^(b-1) is unused), so 2-bit keys take -1, 0, 1.
# * The scale is rounded up to fp16, which keeps |u_tj / s_j| <= Q for the
#   stored scale, hence |u_tj - deq_tj| <= s_j / 2 and no clamp fires.
# * As for the token-wise rule, the integer decision is taken in float32:
#   max |u| / Q is a float32 division, and the code is round-half-even of the
#   exact product u_tj * (1 / s_j) with a float32-rounded reciprocal.
# * A channel with max |u| = 0 gets s = 0 and codes 0.
# * In the page a code is stored as c + 2^(b-1) (offset binary, 1 .. 2^b - 1),
#   packed like the token-wise codes.
# ------------------------------------------------------------------------

def channel_levels(bits: int) -> int:
    """Q = 2^(b-1) - 1, the largest code magnitude of the symmetric quantizer."""
    if bits not in (2, 4, 8):
        raise ValueError(f"unsupported bit-width {bits}")
    return (1 << (bits - 1)) - 1


def channel_scales(u32: np.ndarray, bits: int) -> np.ndarray:
    """fp16 s[..., d] per channel for groups u32[..., n, d] (n tokens each)."""
    u32 = np.asarray(u32, dtype=np.float32)
    amax = np.abs(u32).max(axis=-2)                              # exact
    return fp16.round_up((amax / np.float32(channel_levels(bits))).astype(np.float32))


def channel_codes_given(u32: np.ndarray, s: np.ndarray, bits: int,
                        clip: bool = True) -> np.ndarray:
    """Signed codes int64[..., n, d] of groups u32[..., n, d] for channel scales
    s[..., d] (``clip=False``: the raw rounded values, for the clamp test)."""
    u32 = np.asarray(u32, dtype=np.float32)
    sf = np.asarray(s, dtype=np.float16).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(sf > 0, (np.float32(1.0) / sf).astype(np.float32), np.float32(0.0))
    prod = u32.astype(np.float64) * inv.astype(np.float64)[..., None, :]   # exact product
    c = np.rint(prod).astype(np.int64)                                      # half to even
    c = np.where((sf > 0)[..., None, :], c, 0)
    if clip:
        q = channel_levels(bits)
        c = np.clip(c, -q, q)
    return c


def quantize_channels(u32: np.ndarray, bits: int):
    """(signed codes int64[..., n, d], s fp16[..., d]) for float32 groups."""
    s = channel_scales(u32, bits)
    return channel_codes_given(u32, s, bits), s


def dequantize_channels(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    """deq = c * s (per channel) in float64, codes[..., n, d], s[..., d]."""
    sf = np.asarray(s, dtype=np.float16).astype(np.float64)
    return np.asarray(codes, dtype=np.float64) * sf[..., None, :]

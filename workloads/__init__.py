"""Seeded synthetic inputs shared by the CPU oracle, the tests and the benchmark.

This module only draws numbers: it holds none of the quantizer's, the
rotation's or the attention's arithmetic.  Everything here is deterministic
from a seed (NumPy PCG64).  Floating-point tensors are drawn in float32 and
rounded to bfloat16 with round-to-nearest-even, so that the oracle and the
GPU path see identical bits.

Workload shapes follow the five synthetic configurations this library is
measured on (sizes written out below).  The pages describe real-model KV
caches; these generators stand in for them with the stated distributions:

* values ~ N(0, 1);
* a few "outlier" channels per KV head multiplied by a seeded factor, the
  kind of large-magnitude channels the SAW-INT4 explainer blames for naive
  INT4 failing ("SAW-INT4: System-Aware 4-Bit KV-Cache Quantization ...",
  section 2, "mix before you shrink");
* per-component sensitivities ~ lognormal(0, 1) times a U-shape over depth,
  the shape the RateQuant summary reports for gradient sensitivity
  (RateQuant technical summary, Methodology section 2).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

PAGE_SIZE = 16


# ---------------------------------------------------------------------------
# bfloat16 helpers (input preparation only)
# ---------------------------------------------------------------------------

def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even).

    Returns float32 values that are exactly representable in bfloat16.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) & np.uint32(0xFFFF0000)).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bfloat16-exact."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16)


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    """float32 values from raw bfloat16 bit patterns."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# workload descriptions
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    num_layers: int
    batch: int
    hq: int
    hkv: int
    head_dim: int
    ctx: int                     # tokens per sequence at decode time (incl. window)
    had_block: int
    window: int                  # bf16 residual window R (0 = none)
    k_bits: Optional[int]        # None: set per head by the allocator
    v_bits: Optional[int]
    q_fp32: bool
    k_outliers: int              # outlier channels per KV head in K
    v_outliers: int
    outlier_lo: float
    outlier_hi: float
    new_tokens: int = 0          # append workloads: tokens appended per sequence


TINY = Workload("tiny-correctness", 1001, 1, 1, 4, 4, 64, 256, 64, 0, 4, 2, True,
                2, 2, 20.0, 20.0)
LLAMA3_8B_LAYER = Workload("llama3-8b-decode-layer", 1002, 1, 16, 32, 8, 128, 4096, 128, 0,
                           4, 4, False, 4, 0, 10.0, 50.0)
MIXED_32L = Workload("mixed-bits-32-layers", 1003, 32, 64, 32, 8, 128, 2048, 128, 0,
                     None, None, False, 4, 0, 10.0, 50.0)
LONG_CONTEXT = Workload("long-context-131k", 1004, 1, 1, 32, 8, 128, 131072, 128, 128,
                        4, 2, False, 4, 4, 10.0, 50.0)
APPEND_SWEEP = Workload("append-sweep-8x8192", 1005, 1, 8, 32, 8, 128, 8192, 128, 0,
                        4, 4, False, 4, 4, 10.0, 50.0, new_tokens=8192)

ALL = (TINY, LLAMA3_8B_LAYER, MIXED_32L, LONG_CONTEXT, APPEND_SWEEP)
APPEND_BLOCKS = (32, 64, 128)
APPEND_BITS = (2, 4, 8)


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

def rng_for(seed: int, *stream: int) -> np.random.Generator:
    """Independent PCG64 stream for (seed, *stream)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def outlier_channels(seed: int, hkv: int, d: int, count: int, lo: float, hi: float,
                     stream: int) -> tuple[np.ndarray, np.ndarray]:
    """Seeded outlier channel indices [hkv, count] and their factors [hkv, count]."""
    rng = rng_for(seed, 7, stream)
    idx = np.stack([rng.choice(d, size=count, replace=False) for _ in range(hkv)]) \
        if count else np.zeros((hkv, 0), dtype=np.int64)
    fac = rng.uniform(lo, hi, size=(hkv, count)).astype(np.float32)
    return idx, fac


def kv_tokens(seed: int, stream: int, batch: int, tokens: int, hkv: int, d: int,
              n_outliers: int, lo: float, hi: float, start: int = 0,
              seq0: int = 0) -> np.ndarray:
    """bf16-exact float32 K or V tokens, shape [batch, tokens, hkv, d].

    ``stream`` separates K (0) from V (1) and layers (2*layer + kv).  Token
    ``start`` offsets the draw so that a long sequence can be generated in
    chunks: the values of token t of sequence b do not depend on how the
    sequence is chunked.  The rows are sequences seq0 .. seq0 + batch - 1 of
    the stream (same outlier channels, independent tokens).
    """
    out = np.empty((batch, tokens, hkv, d), dtype=np.float32)
    idx, fac = outlier_channels(seed, hkv, d, n_outliers, lo, hi, stream)
    chunk = 4096
    for b in range(batch):
        t0 = start
        while t0 < start + tokens:
            t1 = min(start + tokens, (t0 // chunk + 1) * chunk)
            rng = rng_for(seed, stream, seq0 + b, t0 // chunk)
            # the generator is sequential: drawing up to t1 gives the prefix of
            # the whole chunk's draw
            block = rng.standard_normal((t1 - (t0 // chunk) * chunk, hkv, d), dtype=np.float32)
            block = block[t0 - (t0 // chunk) * chunk:]
            if n_outliers:
                for h in range(hkv):
                    block[:, h, idx[h]] *= fac[h]
            out[b, t0 - start:t1 - start] = block
            t0 = t1
    return round_to_bf16(out)


def queries(seed: int, stream: int, batch: int, hq: int, d: int, fp32: bool) -> np.ndarray:
    """Decode queries [batch, hq, d] ~ N(0, 1); bf16-exact unless ``fp32``."""
    rng = rng_for(seed, 100 + stream)
    q = rng.standard_normal((batch, hq, d), dtype=np.float32)
    return q if fp32 else round_to_bf16(q)


def page_table(seed: int, batch: int, max_pages: int, num_pages: Optional[int] = None,
               stream: int = 0) -> np.ndarray:
    """int32 [batch, max_pages] page table over a seeded random permutation.

    Every logical page of every sequence gets a distinct physical page, so
    that no two sequences share storage and consecutive logical pages are
    not contiguous in memory.
    """
    total = batch * max_pages
    if num_pages is None:
        num_pages = total
    assert num_pages >= total
    rng = rng_for(seed, 200 + stream)
    perm = rng.permutation(num_pages)[:total].astype(np.int32)
    return perm.reshape(batch, max_pages)


def sensitivities(seed: int, num_layers: int, hkv: int) -> np.ndarray:
    """float64 [num_layers, hkv, 2] (K, V) sensitivities.

    lognormal(0, 1) per component, times U(l) = 1 + 3 (2 l / (L-1) - 1)^2, a
    U-shape over depth: high in early and late layers.
    """
    rng = rng_for(seed, 300)
    w = rng.lognormal(0.0, 1.0, size=(num_layers, hkv, 2))
    denom = max(num_layers - 1, 1)
    u = 1.0 + 3.0 * (2.0 * np.arange(num_layers) / denom - 1.0) ** 2
    return w * u[:, None, None]


def ragged_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    """int32 [batch] sequence lengths drawn uniformly from [lo, hi]."""
    rng = rng_for(seed, 400)
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def pages_for(tokens: int) -> int:
    return (tokens + PAGE_SIZE - 1) // PAGE_SIZE


def describe(w: Workload) -> dict:
    return dataclasses.asdict(w)


__all__ = [
    "PAGE_SIZE", "Workload", "ALL", "TINY", "LLAMA3_8B_LAYER", "MIXED_32L", "LONG_CONTEXT",
    "APPEND_SWEEP", "APPEND_BLOCKS", "APPEND_BITS", "round_to_bf16", "bf16_bits",
    "bf16_from_bits", "rng_for", "outlier_channels", "kv_tokens", "queries", "page_table",
    "sensitivities", "ragged_lengths", "pages_for", "describe",
]

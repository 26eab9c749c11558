"""Decode attention over the dequantized paged cache.

Sources:
* "SAW-INT4 ...", section 3 (fused engine): attention reads the compact
  cache; rotation and quantization are undone on the fly.  This oracle does
  the plain thing instead: it dequantizes every cached vector, undoes the
  rotation by explicit matrix multiply, and runs ordinary softmax attention.
* "LogQuant ...", Methodology section 4 (position-agnostic optimisation):
  attention output does not depend on the order of the (key, value) pairs,
  A V = A_P V_P, so full-precision window tokens and quantized tokens may be
  combined in any order.
* RateQuant technical summary, Methodology section 3: in the key-per-channel
  mode a page's keys are dequantized with one scale per channel.
* CriticalKV technical summary, Methodology (perturbation definition): the L1
  distance between two attention outputs, used here to report quantization
  error.

Readings: scores are (q . k) * softmax_scale with softmax_scale = 1/sqrt(d)
by default; one decode query attends to every cached token of its sequence
(no causal mask); query head h reads KV head h // (Hq / Hkv); the output is
float64 here and float32 on the GPU; a sequence of length 0 yields zeros.
"""
from __future__ import annotations

import numpy as np

from . import layout
from .cache import CacheState, quantized_prefix
from .hadamard import unrotate
from .quantizer import dequantize, dequantize_channels


def softmax_attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray,
                      scale: float) -> np.ndarray:
    """o = softmax(keys q * scale) values for q[G, d], keys/values[T, d] (float64)."""
    q = np.asarray(q, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros((q.shape[0], values.shape[-1]))
    s = (q @ np.asarray(keys, dtype=np.float64).T) * scale        # [G, T]
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ np.asarray(values, dtype=np.float64)


def cached_kv(state: CacheState, layer: int, b: int, h: int, length: int,
              page_table: np.ndarray):
    """Reconstructed (keys, values) float64 [length, d] of (sequence b, KV head h)."""
    kpc = state.key_per_channel
    lq = quantized_prefix(length, state.window, kpc)
    rows = state.ring_rows
    d = state.head_dim
    view = state.view(layer)
    pos = np.arange(lq)
    pages = np.asarray(page_table[b, pos // layout.PAGE_SIZE], dtype=np.int64)
    slots = pos % layout.PAGE_SIZE
    out = []
    for kv in (0, 1):
        if lq and kpc and kv == 0:
            # key-per-channel: each page's codes times its channel scales
            deq = [dequantize_channels(*view.read_key_channels(int(pg), h))
                   for pg in pages[::layout.PAGE_SIZE]]
            rec = unrotate(np.concatenate(deq, axis=0), state.had_block)
        elif lq:
            codes, s, z = view.read(pages, slots, h, kv)
            rec = unrotate(dequantize(codes, s, z), state.had_block)
        else:
            rec = np.zeros((0, d))
        if length > lq:
            wpos = np.arange(lq, length) % rows
            win = state.windows[layer][b, h, kv, wpos].astype(np.float64)
            rec = np.concatenate([rec, win], axis=0)
        out.append(rec)
    return out[0], out[1]


def decode(state: CacheState, layer: int, q: np.ndarray, page_table: np.ndarray,
           seq_lens: np.ndarray, scale: float | None = None,
           pairs: list | None = None) -> np.ndarray:
    """o[B, Hq, d] float64 for queries q[B, Hq, d].

    ``pairs`` optionally restricts the work to a list of (b, kv_head); the
    other rows are left as NaN (used to sample full-size workloads).
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = state.num_kv_heads
    g = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.full((bsz, hq, d), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(bsz) for h in range(hkv)]
    for b, h in todo:
        keys, values = cached_kv(state, layer, b, h, int(seq_lens[b]), page_table)
        o[b, h * g:(h + 1) * g] = softmax_attention(q[b, h * g:(h + 1) * g], keys, values,
                                                    scale)
    return o


def l1_perturbation(o: np.ndarray, o_hat: np.ndarray) -> float:
    """CriticalKV's output perturbation || o - o_hat ||_1 (summed over all rows)."""
    return float(np.abs(np.asarray(o, np.float64) - np.asarray(o_hat, np.float64)).sum())


def exact_decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, seq_lens: np.ndarray,
                 scale: float | None = None, pairs: list | None = None) -> np.ndarray:
    """Unquantized attention o[B, Hq, d] over the original K/V [B, T, Hkv, d]
    (bf16 values widened exactly), the reference the quantization error is
    measured against.  ``pairs`` as in ``decode``."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = k.shape[2]
    g = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.full((bsz, hq, d), np.nan)
    todo = pairs if pairs is not None else [(b, h) for b in range(bsz) for h in range(hkv)]
    for b, h in todo:
        n = int(seq_lens[b])
        o[b, h * g:(h + 1) * g] = softmax_attention(q[b, h * g:(h + 1) * g], k[b, :n, h],
                                                    v[b, :n, h], scale)
    return o


def quant_error(o_hat: np.ndarray, o_ref: np.ndarray) -> dict:
    """Error of attention over the quantized cache (o_hat) against attention
    over the unquantized K/V (o_ref), over the rows o_ref holds (not NaN):
    max and mean absolute difference, the relative L2 norm of the difference
    ||o_hat - o_ref||_2 / ||o_ref||_2, and CriticalKV's L1 perturbation
    ||o_ref - o_hat||_1 per query row (the sum divided by the rows)."""
    o_hat = np.asarray(o_hat, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    rows = ~np.isnan(o_ref).any(axis=-1)
    a, r = o_hat[rows], o_ref[rows]
    diff = a - r
    n = int(rows.sum())
    return {"max_abs": float(np.abs(diff).max()) if n else 0.0,
            "mean_abs": float(np.abs(diff).mean()) if n else 0.0,
            "rel_l2": float(np.linalg.norm(diff) / np.linalg.norm(r)) if n else 0.0,
            "l1_per_row": l1_perturbation(r, a) / n if n else 0.0,
            "rows": n}

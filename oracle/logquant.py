"""LogQuant's log-spaced full-precision selection, and attention with it.

Test infrastructure, like the rest of this package: only the tests and the
bench's CPU baseline use it; the library never imports it.

Source: "LogQuant: Log-Distributed 2-Bit Quantization of KV Cache with
Superior Accuracy Preservation" (technical summary), Methodology section 2
(log-based filtering: a base window W, the most recent tokens kept at full
precision, sparser selections further back, a 3W full-precision reserve, and
the halving of older selections as tokens arrive) and section 4 (A V = A_P V_P:
full-precision and quantized tokens combine in any order).

Reading of section 2 (the summary leaves the bookkeeping open):
* B, the set of positions kept at full precision, starts empty; every
  appended token joins B.
* When |B| reaches 3W, the oldest 2W members of B are halved: of each
  consecutive pair (by position) the first stays and the second leaves B.
  |B| drops to 2W and new tokens fill it again.
* Every token is quantized on arrival; tokens outside B are read from the
  quantized cache, tokens in B use their bf16 values.
Repeated halving keeps, right after a halving, the newest W - 1 positions
one apart, then W / 2 two apart, W / 4 four apart, ..., one W apart, plus
position 0 (the first of every pair it is in).
"""
from __future__ import annotations

import numpy as np

from .attention import cached_kv, softmax_attention
from .cache import CacheState


def members(length: int, w: int) -> np.ndarray:
    """Sorted positions of B after `length` appends with base window w."""
    if w < 1:
        raise ValueError("w must be >= 1")
    b: list[int] = []
    for p in range(length):
        b.append(p)
        if len(b) == 3 * w:
            b = b[0:2 * w:2] + b[2 * w:]
    return np.asarray(b, dtype=np.int64)


def decode(state: CacheState, layer: int, q: np.ndarray, page_table: np.ndarray,
           seq_lens: np.ndarray, w: int, k_bf16: np.ndarray, v_bf16: np.ndarray,
           scale: float | None = None) -> np.ndarray:
    """o[B, Hq, d] float64: attention over the quantized cache (window 0) in
    which the positions of B use the bf16 keys and values k_bf16, v_bf16
    [B][T][Hkv][d] (the appended tokens, bf16-exact floats)."""
    if state.window or state.key_per_channel:
        raise ValueError("the LogQuant reserve replaces the bf16 window: window must be 0, "
                         "keys token-wise")
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = state.num_kv_heads
    g = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((bsz, hq, d))
    for b in range(bsz):
        n = int(seq_lens[b])
        keep = members(n, w)
        for h in range(hkv):
            keys, values = cached_kv(state, layer, b, h, n, page_table)
            keys[keep] = np.asarray(k_bf16[b, keep, h], dtype=np.float64)
            values[keep] = np.asarray(v_bf16[b, keep, h], dtype=np.float64)
            o[b, h * g:(h + 1) * g] = softmax_attention(q[b, h * g:(h + 1) * g], keys, values,
                                                        scale)
    return o

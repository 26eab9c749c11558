"""Quantize-on-append into the paged cache, plus the bf16 recent-token window.

Sources:
* "SAW-INT4 ...", summary and section 2: each new K/V head vector is rotated
  by a block-diagonal Hadamard transform and quantized token-wise; section 1:
  the cache lives in uniform fixed-size pages.
* RateQuant technical summary, Methodology section 3: K and V of every
  (layer, head) are separate components with their own bit-widths
  (the per-layer table ``bits[h] = (bK, bV)``).
* "LogQuant: Log-Distributed 2-Bit Quantization of KV Cache ...",
  Methodology section 2 (window configuration / full-precision reserve): the
  most recent tokens are kept at full precision.

Semantics (readings where the pages are silent):
* Position p of sequence b lives in logical page p // 16 at slot p % 16;
  ``page_table[b, p // 16]`` names the physical page.
* With a window of R > 0 tokens, after an append the last min(L, R)
  positions of a sequence of length L are held as bf16 in a ring indexed by
  p mod R; positions p < L - R are quantized.  A token is quantized when it
  leaves the window (its bf16 value is read from the ring) or directly from
  the appended input if it never enters the window.
* With R = 0 every appended token is quantized.

Key-per-channel mode (RateQuant technical summary, Methodology section 3:
KIVI's symmetric per-channel keys beside asymmetric per-token values;
"LogQuant ...", section 5: key-per-channel):
* A page's keys are quantized together, one fp16 scale per channel
  (``quantizer.quantize_channels``), so a page is quantized only once all of
  its 16 positions have left the window: the quantized prefix of a sequence of
  length L is Q(L) = 16 * floor(max(L - R, 0) / 16), K and V alike (values stay
  token-wise).  Positions Q(L) .. L - 1 (at most R + 15) keep their bf16 K and
  V in a ring of R + 16 rows indexed by p mod (R + 16); with R = 0 the ring
  holds the page still being filled.
* An append quantizes the pages that its new length completes, reading each
  position from the ring (older positions) or from the appended input, then
  writes the new positions that stay in bf16 into the ring.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

from . import layout
from .hadamard import rotate
from .quantizer import quantize, quantize_channels, rotate_and_quantize


@dataclasses.dataclass
class CacheState:
    head_dim: int
    had_block: int
    window: int
    bits: np.ndarray                 # int [L, Hkv, 2]
    pools: List[np.ndarray]          # per layer uint8 [num_pages, page_bytes]
    windows: Optional[List[np.ndarray]]  # per layer float32 [Bmax, Hkv, 2, rows, d] or None
    key_per_channel: bool = False

    @property
    def num_kv_heads(self) -> int:
        return int(self.bits.shape[1])

    @property
    def ring_rows(self) -> int:
        return ring_rows(self.window, self.key_per_channel)

    def view(self, layer: int) -> layout.PageView:
        return layout.PageView(self.pools[layer], self.head_dim, self.bits[layer],
                               self.key_per_channel)


def ring_rows(window: int, key_per_channel: bool = False) -> int:
    """Rows of the bf16 ring per (sequence, KV head, K|V)."""
    return window + layout.PAGE_SIZE if key_per_channel else window


def quantized_prefix(length: int, window: int, key_per_channel: bool = False) -> int:
    """Positions 0 .. Q - 1 of a sequence of this length are quantized."""
    if key_per_channel:
        return layout.PAGE_SIZE * (max(0, length - window) // layout.PAGE_SIZE)
    return max(0, length - window) if window else length


def new_state(num_layers: int, num_pages: int, head_dim: int, had_block: int,
              bits: np.ndarray, window: int = 0, max_batch: int = 0,
              key_per_channel: bool = False) -> CacheState:
    bits = np.asarray(bits, dtype=np.int64).reshape(num_layers, -1, 2)
    hkv = bits.shape[1]
    pools = [np.zeros((num_pages, layout.page_bytes(head_dim, bits[l], key_per_channel)),
                      dtype=np.uint8) for l in range(num_layers)]
    wins = None
    rows = ring_rows(window, key_per_channel)
    if rows:
        wins = [np.zeros((max_batch, hkv, 2, rows, head_dim), dtype=np.float32)
                for _ in range(num_layers)]
    return CacheState(head_dim, had_block, window, bits, pools, wins, key_per_channel)


def append(state: CacheState, layer: int, k: np.ndarray, v: np.ndarray,
           page_table: np.ndarray, seq_lens: np.ndarray, window_row: int = 0) -> dict:
    """Append k, v [B, T_new, Hkv, d] (bf16-exact float32) after seq_lens[b] tokens.

    Sequence b of the call uses window row window_row + b (its page-table row is
    page_table[b]).

    Mutates ``state`` and returns, for tests, a dict keyed by (b, h, kv) of
    (positions, codes, s, z, u32): the positions quantized by this call, what
    was written for them, and the float32-rounded rotated vectors.
    """
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    if state.key_per_channel:
        return _append_key_channels(state, layer, k, v, page_table, seq_lens, window_row)
    bsz, t_new, hkv, d = k.shape
    r = state.window
    view = state.view(layer)
    written = {}
    for b in range(bsz):
        l0 = int(seq_lens[b])
        l_end = l0 + t_new
        q_old = max(0, l0 - r) if r else l0
        q_new = max(0, l_end - r) if r else l_end
        pos = np.arange(q_old, q_new)
        from_ring = pos < l0                  # leaving the window: bf16 value in the ring
        for kv, src in ((0, k), (1, v)):
            for h in range(hkv):
                if not len(pos):
                    continue
                bits = int(state.bits[layer, h, kv])
                vecs = np.empty((len(pos), d), dtype=np.float32)
                if from_ring.any():
                    vecs[from_ring] = state.windows[layer][window_row + b, h, kv, pos[from_ring] % r]
                if (~from_ring).any():
                    vecs[~from_ring] = src[b, pos[~from_ring] - l0, h]
                codes, s, z, u32 = rotate_and_quantize(vecs, state.had_block, bits)
                pages = np.asarray(page_table[b, pos // layout.PAGE_SIZE], dtype=np.int64)
                view.write_many(pages, pos % layout.PAGE_SIZE, h, kv, codes, s, z)
                written[(b, h, kv)] = (pos, codes, s, z, u32)
        if r:
            for p in range(max(l0, q_new), l_end):
                state.windows[layer][window_row + b, :, 0, p % r] = k[b, p - l0]
                state.windows[layer][window_row + b, :, 1, p % r] = v[b, p - l0]
    return written


def _append_key_channels(state: CacheState, layer: int, k: np.ndarray, v: np.ndarray,
                         page_table: np.ndarray, seq_lens: np.ndarray,
                         window_row: int) -> dict:
    """``append`` in the key-per-channel mode (see the module docstring).

    Returns, keyed by (b, h, kv), (positions, codes, scales, zeros, u32) of the
    pages it quantized: for K the signed codes [n, d] and the channel scales
    [pages, d] (zeros None), for V as in ``append``."""
    bsz, t_new, hkv, d = k.shape
    r = state.window
    rows = state.ring_rows
    ring = state.windows[layer]
    view = state.view(layer)
    ps = layout.PAGE_SIZE
    written = {}
    for b in range(bsz):
        l0 = int(seq_lens[b])
        l_end = l0 + t_new
        q_old = quantized_prefix(l0, r, True)
        q_new = quantized_prefix(l_end, r, True)
        pos = np.arange(q_old, q_new)
        from_ring = pos < l0
        for kv, src in ((0, k), (1, v)):
            for h in range(hkv):
                if not len(pos):
                    continue
                bits = int(state.bits[layer, h, kv])
                vecs = np.empty((len(pos), d), dtype=np.float32)
                if from_ring.any():
                    vecs[from_ring] = ring[window_row + b, h, kv, pos[from_ring] % rows]
                if (~from_ring).any():
                    vecs[~from_ring] = src[b, pos[~from_ring] - l0, h]
                u32 = rotate(vecs, state.had_block).astype(np.float32)
                pages = np.asarray(page_table[b, pos[::ps] // ps], dtype=np.int64)
                if kv == 0:
                    groups = u32.reshape(-1, ps, d)
                    codes, s = quantize_channels(groups, bits)
                    for i, pg in enumerate(pages):
                        view.write_key_channels(int(pg), h, codes[i], s[i])
                    written[(b, h, kv)] = (pos, codes.reshape(-1, d), s, None, u32)
                else:
                    codes, s, z = quantize(u32, bits)
                    view.write_many(np.repeat(pages, ps), pos % ps, h, kv, codes, s, z)
                    written[(b, h, kv)] = (pos, codes, s, z, u32)
        for p in range(max(l0, q_new), l_end):
            ring[window_row + b, :, 0, p % rows] = k[b, p - l0]
            ring[window_row + b, :, 1, p % rows] = v[b, p - l0]
    return written

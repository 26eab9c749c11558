"""Byte layout of one page of the paged quantized KV cache.

Source for the structure: "SAW-INT4 ...", section 1 (the serving system's
paged attention stores the cache in uniform fixed-size blocks, which is why
token eviction is hard and token-wise quantization fits).  The byte layout
inside a page is a convention of this library (the pages do not give one):

A page holds PAGE_SIZE = 16 consecutive token positions of one sequence for
every KV head of one layer.  For each KV head h, in order h = 0 .. Hkv-1, a
contiguous segment of

    K codes   [16][d * bK / 8]   token-major, packed little-endian in bytes
    V codes   [16][d * bV / 8]
    K (s, z)  [16] x 2 x fp16     s first, then z
    V (s, z)  [16] x 2 x fp16

Codes are packed with element j at bit offset (j * b) mod 8 of byte
(j * b) // 8, i.e. for 4-bit codes element 2i is the low nibble of byte i.
Every segment is a multiple of 16 bytes.

In the key-per-channel mode the K (s, z) pairs give way to one fp16 scale per
channel of the page's keys, and the K codes are stored in offset binary
(c + 2^(b-1)):

    K codes   [16][d * bK / 8]
    V codes   [16][d * bV / 8]
    K scales  [d] x fp16         channel j's scale for the page's 16 keys
    V (s, z)  [16] x 2 x fp16
"""
from __future__ import annotations

import numpy as np

PAGE_SIZE = 16


def head_bytes(d: int, bk: int, bv: int, kpc: bool = False) -> int:
    if kpc:
        return PAGE_SIZE * (d * bk // 8 + d * bv // 8) + 2 * d + PAGE_SIZE * 4
    return PAGE_SIZE * (d * bk // 8 + d * bv // 8 + 8)


def head_offsets(d: int, bits: np.ndarray, kpc: bool = False) -> np.ndarray:
    """Byte offset of each head's segment in a page; bits: int[Hkv, 2]."""
    sizes = [head_bytes(d, int(b[0]), int(b[1]), kpc) for b in bits]
    return np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)


def page_bytes(d: int, bits: np.ndarray, kpc: bool = False) -> int:
    return int(sum(head_bytes(d, int(b[0]), int(b[1]), kpc) for b in bits))


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack codes[..., d] (values < 2^bits) into uint8[..., d * bits / 8]."""
    c = np.asarray(codes, dtype=np.uint8)
    per = 8 // bits
    d = c.shape[-1]
    c = c.reshape(*c.shape[:-1], d // per, per).astype(np.uint16)
    shifts = (np.arange(per) * bits).astype(np.uint16)
    return (c << shifts).sum(axis=-1).astype(np.uint8)


def unpack(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    """Inverse of ``pack``: uint8[..., d * bits / 8] -> uint8[..., d]."""
    p = np.asarray(packed, dtype=np.uint8)
    per = 8 // bits
    shifts = (np.arange(per) * bits).astype(np.uint8)
    mask = np.uint8((1 << bits) - 1)
    c = (p[..., None] >> shifts) & mask
    return c.reshape(*p.shape[:-1], d)


class PageView:
    """Field accessors for one layer's pool: uint8[num_pages, page_bytes]."""

    def __init__(self, pool: np.ndarray, d: int, bits: np.ndarray, kpc: bool = False):
        self.pool = pool
        self.d = d
        self.bits = np.asarray(bits, dtype=np.int64)
        self.kpc = kpc
        self.off = head_offsets(d, self.bits, kpc)

    def _seg(self, h: int):
        """(bK, bV, K codes, V codes, K (s, z) or K scales, V (s, z)) offsets."""
        d = self.d
        bk, bv = int(self.bits[h, 0]), int(self.bits[h, 1])
        o = int(self.off[h])
        kc = o
        vc = kc + PAGE_SIZE * d * bk // 8
        ksz = vc + PAGE_SIZE * d * bv // 8
        vsz = ksz + (2 * d if self.kpc else PAGE_SIZE * 4)
        return bk, bv, kc, vc, ksz, vsz

    def read_key_channels(self, page: int, h: int):
        """Key-per-channel mode: (signed codes int64[16, d], scales fp16[d]) of
        one page of head h."""
        d = self.d
        bk, _, kc, _, ksc, _ = self._seg(h)
        nb = d * bk // 8
        packed = self.pool[page, kc:kc + PAGE_SIZE * nb].reshape(PAGE_SIZE, nb)
        codes = unpack(packed, bk, d).astype(np.int64) - (1 << (bk - 1))
        s = self.pool[page, ksc:ksc + 2 * d].copy().view(np.float16)
        return codes, s

    def write_key_channels(self, page: int, h: int, codes: np.ndarray, s: np.ndarray) -> None:
        """Key-per-channel mode: store signed codes[16, d] and scales s[d]."""
        d = self.d
        bk, _, kc, _, ksc, _ = self._seg(h)
        nb = d * bk // 8
        stored = np.asarray(codes, np.int64) + (1 << (bk - 1))
        self.pool[page, kc:kc + PAGE_SIZE * nb] = pack(stored, bk).reshape(-1)
        self.pool[page, ksc:ksc + 2 * d] = np.asarray(s, np.float16).view(np.uint8)

    def read(self, page: np.ndarray, slot: np.ndarray, h: int, kv: int):
        """(codes uint8[n, d], s fp16[n], z fp16[n]) for arrays of pages/slots."""
        d = self.d
        bk, bv, kc, vc, ksz, vsz = self._seg(h)
        if self.kpc and kv == 0:
            raise ValueError("key-per-channel pages: use read/write_key_channels for K")
        b, cbase, sbase = (bk, kc, ksz) if kv == 0 else (bv, vc, vsz)
        nb = d * b // 8
        page = np.asarray(page, dtype=np.int64)
        slot = np.asarray(slot, dtype=np.int64)
        cols = cbase + slot[:, None] * nb + np.arange(nb)[None, :]
        packed = self.pool[page[:, None], cols]
        codes = unpack(packed, b, d)
        scol = sbase + slot[:, None] * 4 + np.arange(4)[None, :]
        sz = self.pool[page[:, None], scol].copy().view(np.float16).reshape(-1, 2)
        return codes, sz[:, 0].copy(), sz[:, 1].copy()

    def write(self, page: int, slot: int, h: int, kv: int, codes: np.ndarray,
              s: np.float16, z: np.float16) -> None:
        d = self.d
        bk, bv, kc, vc, ksz, vsz = self._seg(h)
        if self.kpc and kv == 0:
            raise ValueError("key-per-channel pages: use read/write_key_channels for K")
        b, cbase, sbase = (bk, kc, ksz) if kv == 0 else (bv, vc, vsz)
        nb = d * b // 8
        self.pool[page, cbase + slot * nb: cbase + (slot + 1) * nb] = pack(codes, b)
        sz = np.array([s, z], dtype=np.float16).view(np.uint8)
        self.pool[page, sbase + slot * 4: sbase + slot * 4 + 4] = sz

    def write_many(self, pages: np.ndarray, slots: np.ndarray, h: int, kv: int,
                   codes: np.ndarray, s: np.ndarray, z: np.ndarray) -> None:
        """Vectorised ``write`` for arrays of pages/slots and codes[n, d]."""
        d = self.d
        bk, bv, kc, vc, ksz, vsz = self._seg(h)
        if self.kpc and kv == 0:
            raise ValueError("key-per-channel pages: use read/write_key_channels for K")
        b, cbase, sbase = (bk, kc, ksz) if kv == 0 else (bv, vc, vsz)
        nb = d * b // 8
        pages = np.asarray(pages, dtype=np.int64)
        slots = np.asarray(slots, dtype=np.int64)
        cols = cbase + slots[:, None] * nb + np.arange(nb)[None, :]
        self.pool[pages[:, None], cols] = pack(codes, b)
        sz = np.stack([np.asarray(s, np.float16), np.asarray(z, np.float16)], axis=1)
        scol = sbase + slots[:, None] * 4 + np.arange(4)[None, :]
        self.pool[pages[:, None], scol] = sz.view(np.uint8).reshape(-1, 4)

"""Comparison rules between the CUDA path and the oracle.

Codes and scale/zero ("bit-exact except at rounding boundaries"):
  * (s, z) of a vector must equal the oracle's, except at fp16 rounding
    boundaries: z may differ when the oracle's min lies within 1e-6
    (relative) of an fp16 grid point, and s must then equal the oracle's rule
    applied to the GPU's z, except when that quotient lies within 1e-6 of a
    grid point.  (The GPU computes the rotation with fp32 butterflies, the
    oracle exactly, so values that sit on a rounding boundary may fall
    either way.)
  * Given the GPU's (s, z), each code must equal the oracle's decision
    round-half-even((u - z) / s) except by +-1 where the oracle's quotient t
    lies within 1e-6 * (|u| + |z|) / s of a half-integer (the relative
    rounding error of u and z, carried into units of codes); such flips must
    be fewer than 1e-5 of all codes (a sample of fewer than 1e5 codes may
    hold one).
Per-channel keys (key-per-channel mode): the channel scale and the signed
codes by the same boundary rules (compare_key_channels).
Attention outputs: max |o_gpu - o_oracle| <= 2e-3 and mean <= 2e-4 (fp32
accumulation), with the oracle run over the GPU-written cache.
"""
from __future__ import annotations

import numpy as np

from oracle import fp16, layout, quantizer

CODE_REL = 1e-6
FLIP_FRACTION = 1e-5
O_MAX_ABS = 2e-3
O_MEAN_ABS = 2e-4


def _near_fp16_boundary(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float64)
    lo = fp16.round_down(x).astype(np.float64)
    hi = fp16.round_up(x).astype(np.float64)
    dist = np.minimum(np.abs(x - lo), np.abs(hi - x))
    return dist <= CODE_REL * np.abs(x)


def compare_written(gpu_pool: np.ndarray, written: dict, page_table: np.ndarray, d: int,
                    bits: np.ndarray, kpc: bool = False) -> dict:
    """Check what the GPU wrote for every (b, h, kv) the oracle append wrote
    (in the key-per-channel mode: the values; the keys go to
    compare_key_channels)."""
    view = layout.PageView(gpu_pool, d, bits, kpc)
    if kpc:
        written = {key: val for key, val in written.items() if key[2] == 1}
    stats = dict(vectors=0, codes=0, flips=0, sz_boundary=0)
    for (b, h, kv), (pos, codes, s, z, u32) in written.items():
        if len(pos) == 0:
            continue
        b_ = int(bits[h, kv])
        pages = np.asarray(page_table[b, pos // 16], np.int64)
        gc, gs, gz = view.read(pages, pos % 16, h, kv)
        same = (gs.view(np.uint16) == s.view(np.uint16)) & (gz.view(np.uint16) == z.view(np.uint16))
        if not same.all():
            bad = np.nonzero(~same)[0]
            m = np.float32((1 << b_) - 1)
            mn = u32[bad].min(axis=1)
            z_ok = (gz[bad].view(np.uint16) == z[bad].view(np.uint16)) | _near_fp16_boundary(mn)
            # s follows from the GPU's z: the oracle's rule applied to that z
            span = (u32[bad].max(axis=1) - gz[bad].astype(np.float32)).astype(np.float32)
            q = (span / m).astype(np.float32)
            s_exp = fp16.round_up(q)
            s_ok = (gs[bad].view(np.uint16) == s_exp.view(np.uint16)) | _near_fp16_boundary(q)
            assert (z_ok & s_ok).all(), (
                f"(s, z) mismatch away from an fp16 boundary at b={b} h={h} kv={kv} "
                f"pos={pos[bad][~(z_ok & s_ok)][:5]}")
            stats["sz_boundary"] += int(len(bad))
        want = quantizer.codes_given(u32, gs, gz, b_).astype(np.int64)
        diff = gc.astype(np.int64) - want
        stats["vectors"] += len(pos)
        stats["codes"] += diff.size
        if diff.any():
            rows, cols = np.nonzero(diff)
            assert np.all(np.abs(diff[rows, cols]) == 1), "code differs by more than 1"
            sf = gs[rows].astype(np.float64)
            zf = gz[rows].astype(np.float64)
            u = u32[rows, cols].astype(np.float64)
            t = (u - zf) / sf
            band = CODE_REL * (np.abs(u) + np.abs(zf)) / sf
            assert np.all(np.abs(np.abs(t - np.floor(t)) - 0.5) <= band), (
                f"code flip away from a rounding boundary at b={b} h={h} kv={kv}")
            stats["flips"] += len(rows)
    if stats["codes"]:
        # the fraction bar is statistical: a small sample may hold one boundary flip
        assert stats["flips"] <= max(1.0, FLIP_FRACTION * stats["codes"]), stats
    return stats


def compare_outputs(o_gpu: np.ndarray, o_ref: np.ndarray, rows=None) -> dict:
    """max / mean absolute difference over the rows the oracle computed."""
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    mask = ~np.isnan(o_ref)
    diff = np.abs(o_gpu[mask] - o_ref[mask])
    stats = dict(max_abs=float(diff.max()) if diff.size else 0.0,
                 mean_abs=float(diff.mean()) if diff.size else 0.0, n=int(diff.size))
    assert np.isfinite(o_gpu[mask]).all(), "non-finite GPU output"
    assert stats["max_abs"] <= O_MAX_ABS, stats
    assert stats["mean_abs"] <= O_MEAN_ABS, stats
    return stats


def compare_key_channels(gpu_pool: np.ndarray, written: dict, page_table: np.ndarray, d: int,
                         bits: np.ndarray) -> dict:
    """Key-per-channel mode: the GPU's channel scales and signed key codes of
    every page the oracle append quantized, by the same rules as the token-wise
    codes -- the scale bit-exact except where max |u| / Q lies within 1e-6 of an
    fp16 grid point, and, given the GPU's scale, each code equal to
    round-half-even(u / s) except by +-1 within the 1e-6 band of a half-integer."""
    view = layout.PageView(gpu_pool, d, bits, kpc=True)
    stats = dict(pages=0, codes=0, flips=0, s_boundary=0)
    for (b, h, kv), (pos, codes, s, _, u32) in written.items():
        if kv != 0 or len(pos) == 0:
            continue
        b_ = int(bits[h, 0])
        q = np.float32(quantizer.channel_levels(b_))
        groups = u32.reshape(-1, 16, d)
        for i, p0 in enumerate(pos[::16]):
            pg = int(page_table[b, p0 // 16])
            gc, gs = view.read_key_channels(pg, h)
            g = groups[i]
            same = gs.view(np.uint16) == s[i].view(np.uint16)
            if not same.all():
                quo = (np.abs(g).max(axis=0) / q).astype(np.float32)
                assert _near_fp16_boundary(quo[~same]).all(), (
                    f"channel scale mismatch away from an fp16 boundary at b={b} h={h} "
                    f"page {p0 // 16} channels {np.nonzero(~same)[0][:5]}")
                stats["s_boundary"] += int((~same).sum())
            want = quantizer.channel_codes_given(g, gs, b_)
            diff = gc - want
            stats["pages"] += 1
            stats["codes"] += diff.size
            if diff.any():
                rows, cols = np.nonzero(diff)
                assert np.all(np.abs(diff[rows, cols]) == 1), "key code differs by more than 1"
                t = g[rows, cols].astype(np.float64) / gs[cols].astype(np.float64)
                band = CODE_REL * np.abs(t)
                assert np.all(np.abs(np.abs(t - np.floor(t)) - 0.5) <= band + 1e-12), (
                    f"key code flip away from a rounding boundary at b={b} h={h}")
                stats["flips"] += len(rows)
    if stats["codes"]:
        assert stats["flips"] <= max(1.0, FLIP_FRACTION * stats["codes"]), stats
    return stats

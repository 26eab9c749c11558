"""Pin of the oracle's integer decision rule against the plain definition.

The quantizer's definition (SAW-INT4 page, summary: token-wise asymmetric
INT-b after a block-diagonal Hadamard rotation; RateQuant technical summary,
Methodology section 3: asymmetric per-token quantization) is, in exact
arithmetic,

    z = fp16_down(min u),  s = fp16_up((max u - z) / M),  c = rint((u - z) / s)

with u the exact rotation.  The oracle takes the same decision in the
kernel's precision instead (u rounded once to fp32, fp32 subtract, fp32
reciprocal, round-half-even of the exact product).  These tests run both
rules on the workloads' own data and require that they disagree only where
the plain rule's quotient sits within the 1e-6 relative band of a rounding
boundary (a half-integer for codes, an fp16 grid point for s and z) -- the
same band within which a code may flip between the GPU and the oracle.  The
counts of such boundary cases are printed (``pytest -s``).  They are not held
to the 1e-5 flip fraction: at 8 bits the fp32 rounding of u and of 1/s moves
4e-5 to 1.3e-4 of the codes across a half-integer, which is why both sides
take the decision in the same (fp32) precision.

A second test drives the fp32 rule through extreme spans (span / M exactly
representable in fp16, subnormal scales, huge ranges) and checks that its
unclipped codes never leave [0, M]: the kernels round codes without a clamp,
which is safe only because the directed rounding of s and z keeps every
quotient at most M + 1/2 - (a margin).
"""
import numpy as np
import pytest

from oracle import fp16, hadamard, quantizer
from workloads import APPEND_SWEEP, LLAMA3_8B_LAYER, kv_tokens

BAND = 1e-6


def _plain_float64(u64: np.ndarray, bits: int):
    """The definition in float64: (codes, s, z) from the exact rotation u64."""
    m = float((1 << bits) - 1)
    z = fp16.round_down(u64.min(axis=-1))
    zf = z.astype(np.float64)
    s = fp16.round_up((u64.max(axis=-1) - zf) / m)
    sf = s.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(sf[:, None] > 0, (u64 - zf[:, None]) / sf[:, None], 0.0)
    return np.rint(t), s, z, t


def _near_grid(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float64)
    lo = fp16.round_down(x).astype(np.float64)
    hi = fp16.round_up(x).astype(np.float64)
    return np.minimum(x - lo, hi - x) <= BAND * np.abs(x)


def _compare(x: np.ndarray, block: int, bits: int) -> dict:
    """Both rules on bf16 vectors x[n, d]; asserts and returns the counts."""
    u64 = hadamard.rotate(x, block)                  # exact: bf16 inputs, +-1 sums
    c64, s64, z64, t = _plain_float64(u64, bits)
    u32 = u64.astype(np.float32)
    s32, z32 = quantizer.scale_zero(u32, bits)
    c32 = quantizer.codes_given(u32, s32, z32, bits)
    m = (1 << bits) - 1
    # (s, z): equal unless min u, or the span quotient, lies on an fp16 boundary
    sz_diff = (s32.view(np.uint16) != s64.view(np.uint16)) | \
              (z32.view(np.uint16) != z64.view(np.uint16))
    zq = (u64.max(axis=-1) - z64.astype(np.float64)) / m
    assert np.all(_near_grid(u64.min(axis=-1))[sz_diff] | _near_grid(zq)[sz_diff]), \
        "(s, z) differ away from an fp16 boundary"
    same = ~sz_diff
    diff = (c32[same] != c64[same])
    # codes: equal unless the plain quotient lies within the band of a half-integer
    tt = t[same][diff]
    uu = u64[same][diff]
    zz = np.broadcast_to(z64[same][:, None].astype(np.float64), c64[same].shape)[diff]
    ss = np.broadcast_to(s64[same][:, None].astype(np.float64), c64[same].shape)[diff]
    assert np.all(np.abs(c32[same][diff] - c64[same][diff]) == 1)
    band = BAND * (np.abs(uu) + np.abs(zz)) / ss
    assert np.all(np.abs(np.abs(tt - np.floor(tt)) - 0.5) <= band), \
        "a code differs away from a rounding boundary"
    return dict(vectors=int(x.shape[0]), codes=int(c64.size), sz_boundary=int(sz_diff.sum()),
                code_flips=int(diff.sum()))


def _c2_vectors():
    w = LLAMA3_8B_LAYER
    out = {}
    for kv, outl in ((0, w.k_outliers), (1, w.v_outliers)):
        x = kv_tokens(w.seed, kv, 2, w.ctx, w.hkv, w.head_dim, outl, w.outlier_lo, w.outlier_hi)
        out[kv] = x.reshape(-1, w.head_dim)
    return out


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_rule_matches_plain_definition_c2(bits):
    """2 of the 16 sequences of the Llama-3-8B-shaped layer (8192 tokens x 8 KV
    heads, K with outlier channels), Hadamard block 128."""
    data = _c2_vectors()
    for kv in (0, 1):
        st = _compare(data[kv], LLAMA3_8B_LAYER.had_block, bits)
        print(f"C2 kv={kv} bits={bits}: {st}")


@pytest.mark.parametrize("block", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_rule_matches_plain_definition_append_sweep(block, bits):
    """One of the 8 sequences of the append sweep (8192 tokens x 8 KV heads, K
    and V with outlier channels) at every (block, bits) point."""
    w = APPEND_SWEEP
    for kv in (0, 1):
        x = kv_tokens(w.seed, kv, 1, w.new_tokens, w.hkv, w.head_dim, w.k_outliers,
                      w.outlier_lo, w.outlier_hi).reshape(-1, w.head_dim)
        st = _compare(x, block, bits)
        print(f"C5 block={block} kv={kv} bits={bits}: {st}")


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_unclipped_codes_stay_in_range_at_extreme_spans(bits):
    m = (1 << bits) - 1
    rng = np.random.default_rng(17 + bits)
    rows = []
    # span / M exactly an fp16 value (the tightest case for s = fp16_up(span / M))
    for e in range(-24, 16):
        s = np.float32(2.0 ** e)
        for k in (1, 3, 7, 1023):
            step = np.float32(s * k / 1024) if e > -14 else s
            z = np.float32(fp16.round_down(np.float64(rng.normal()) * 2.0 ** e))
            span = np.float32(step * m)
            v = z + span * rng.random(64).astype(np.float32)
            v[0], v[1] = z, z + span
            rows.append(v.astype(np.float32))
    # huge, tiny and subnormal ranges with random interior points
    for lo, hi in ((-6e4, 6e4), (-1e-7, 1e-7), (3e-8, 5e-8), (-65000.0, -64000.0),
                   (1000.0, 1000.5)):
        v = rng.uniform(lo, hi, 64).astype(np.float32)
        v[0], v[1] = lo, hi
        rows.append(v)
    u = np.stack(rows)
    s, z = quantizer.scale_zero(u, bits)
    ok = np.isfinite(s.astype(np.float32)) & np.isfinite(z.astype(np.float32))
    raw = quantizer.codes_given(u[ok], s[ok], z[ok], bits, clip=False)
    assert raw.min() >= 0 and raw.max() <= m

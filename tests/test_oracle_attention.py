"""Pins for oracle.attention: brute force, closed forms, invariances, error ordering."""
import math

import numpy as np
import pytest

from oracle import attention, cache, hadamard, layout, quantizer
from workloads import kv_tokens, page_table, queries


def test_softmax_attention_brute_force():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((3, 5))
    k = rng.standard_normal((7, 5))
    v = rng.standard_normal((7, 4))
    got = attention.softmax_attention(q, k, v, 0.4)
    for g in range(3):
        sc = [sum(q[g, i] * k[t, i] for i in range(5)) * 0.4 for t in range(7)]
        e = [math.exp(x) for x in sc]
        for j in range(4):
            assert abs(got[g, j] - sum(e[t] * v[t, j] for t in range(7)) / sum(e)) < 1e-12


def test_two_token_closed_form():
    q = np.array([[1.0, 0.0]])
    k = np.array([[1.0, 0.0], [0.0, 1.0]])
    v = np.array([[1.0, 2.0], [3.0, 4.0]])
    e = math.e
    want = [(e * 1 + 3) / (e + 1), (e * 2 + 4) / (e + 1)]
    assert np.allclose(attention.softmax_attention(q, k, v, 1.0)[0], want, atol=1e-15)


def _filled(bsz, n, hkv, d, block, bits, window, seed=5, outl=4):
    k = kv_tokens(seed, 0, bsz, n, hkv, d, outl, 10.0, 50.0)
    v = kv_tokens(seed, 1, bsz, n, hkv, d, outl, 10.0, 50.0)
    pages = (n + 15) // 16
    pt = page_table(seed, bsz, pages)
    st = cache.new_state(1, bsz * pages, d, block, np.array([[bits] * hkv]), window, bsz)
    cache.append(st, 0, k, v, pt, np.zeros(bsz, np.int32))
    return st, k, v, pt


def test_window_covering_everything_is_exact_bf16_attention():
    st, k, v, pt = _filled(2, 37, 2, 64, 64, (4, 2), window=64)
    q = queries(5, 0, 2, 4, 64, True)
    o = attention.decode(st, 0, q, pt, np.array([37, 37]))
    for b in range(2):
        for h in range(4):
            want = attention.softmax_attention(q[b, h:h + 1], k[b, :, h // 2], v[b, :, h // 2],
                                               1 / 8)
            assert np.allclose(o[b, h], want[0], atol=1e-13)


def test_single_token_returns_the_dequantized_value():
    st, k, v, pt = _filled(1, 1, 1, 64, 64, (4, 4), window=0)
    q = queries(5, 0, 1, 1, 64, True)
    o = attention.decode(st, 0, q, pt, np.array([1]))
    u = hadamard.rotate(v[0, 0, 0], 64).astype(np.float32)[None]
    c, s, z = quantizer.quantize(u, 4)
    want = hadamard.unrotate(quantizer.dequantize(c, s, z), 64)[0]
    assert np.allclose(o[0, 0], want, atol=1e-12)


def test_equal_keys_give_the_mean_value():
    d, n = 64, 20
    st = cache.new_state(1, 4, d, 64, np.array([[[4, 4]]]), 0, 1)
    k = np.tile(kv_tokens(6, 0, 1, 1, 1, d, 0, 1, 1), (1, n, 1, 1))
    v = kv_tokens(6, 1, 1, n, 1, d, 0, 1, 1)
    pt = np.arange(4, dtype=np.int32)[None]
    cache.append(st, 0, k, v, pt, np.zeros(1, np.int32))
    q = queries(6, 0, 1, 1, d, True)
    o = attention.decode(st, 0, q, pt, np.array([n]))
    _, vals = attention.cached_kv(st, 0, 0, 0, n, pt)
    assert np.allclose(o[0, 0], vals.mean(0), atol=1e-12)


def test_permutation_invariance():
    # "LogQuant", Methodology section 4: A V = A_P V_P.
    bsz, n, d = 1, 64, 64
    k = kv_tokens(8, 0, bsz, n, 1, d, 2, 10, 20)
    v = kv_tokens(8, 1, bsz, n, 1, d, 2, 10, 20)
    q = queries(8, 0, 1, 1, d, True)
    outs = []
    for perm_seed in (0, 1):
        perm = np.random.default_rng(perm_seed).permutation(n) if perm_seed else np.arange(n)
        pt = page_table(9 + perm_seed, bsz, 4)
        st = cache.new_state(1, 4, d, 64, np.array([[[4, 2]]]), 0, 1)
        cache.append(st, 0, k[:, perm], v[:, perm], pt, np.zeros(1, np.int32))
        outs.append(attention.decode(st, 0, q, pt, np.array([n])))
    assert np.allclose(outs[0], outs[1], atol=1e-12)


def test_gqa_head_mapping():
    st, k, v, pt = _filled(1, 48, 2, 64, 64, (8, 8), window=0)
    q = queries(5, 1, 1, 8, 64, True)
    o = attention.decode(st, 0, q, pt, np.array([48]))
    for h in range(8):
        kk, vv = attention.cached_kv(st, 0, 0, h // 4, 48, pt)
        want = attention.softmax_attention(q[0, h:h + 1], kk, vv, 1 / 8)[0]
        assert np.allclose(o[0, h], want, atol=1e-13)
        other, vo = attention.cached_kv(st, 0, 0, 1 - h // 4, 48, pt)
        assert not np.allclose(o[0, h], attention.softmax_attention(q[0, h:h + 1], other, vo,
                                                                   1 / 8)[0], atol=1e-3)


def test_error_shrinks_with_bits():
    n, d = 256, 64
    q = queries(10, 0, 1, 4, d, True)
    errs = []
    for bits in ((2, 2), (4, 4), (8, 8)):
        st, k, v, pt = _filled(1, n, 2, d, 64, bits, 0, seed=10)
        o = attention.decode(st, 0, q, pt, np.array([n]))
        ref = np.stack([attention.softmax_attention(q[0, h:h + 1], k[0, :, h // 2],
                                                    v[0, :, h // 2], 1 / 8)[0] for h in range(4)])
        errs.append(np.abs(o[0] - ref).mean())
    assert errs[2] < errs[1] / 8 and errs[1] < errs[0] / 2


def test_empty_sequence_gives_zeros():
    st, k, v, pt = _filled(1, 16, 1, 64, 64, (4, 4), window=0)
    o = attention.decode(st, 0, queries(1, 0, 1, 1, 64, True), pt, np.array([0]))
    assert np.array_equal(o, np.zeros_like(o))


def test_exact_decode_equals_a_window_covering_everything():
    """exact_decode is attention over the bf16 K/V themselves: the same as the
    cache's attention when the bf16 window holds every token."""
    st, k, v, pt = _filled(2, 37, 2, 64, 64, (4, 2), window=64)
    q = queries(5, 2, 2, 4, 64, True)
    lens = np.array([37, 20])
    st2, _, _, _ = _filled(2, 37, 2, 64, 64, (4, 2), window=64)
    want = attention.decode(st, 0, q, pt, np.array([37, 37]))
    got = attention.exact_decode(q, k, v, np.array([37, 37]))
    assert np.allclose(got, want, atol=1e-13)
    part = attention.exact_decode(q, k, v, lens, pairs=[(1, 0)])
    assert np.isnan(part[0]).all() and np.isnan(part[1, 2:]).all()
    ref = attention.softmax_attention(q[1, :2], k[1, :20, 0], v[1, :20, 0], 1 / 8)
    assert np.allclose(part[1, :2], ref, atol=1e-14)


def test_quant_error_closed_form():
    o_ref = np.array([[[3.0, 4.0], [np.nan, np.nan]], [[0.0, 1.0], [1.0, 0.0]]])
    o_hat = np.array([[[3.0, 5.0], [9.0, 9.0]], [[-1.0, 1.0], [1.0, 0.0]]])
    e = attention.quant_error(o_hat, o_ref)
    assert e["rows"] == 3
    assert e["max_abs"] == 1.0
    assert abs(e["mean_abs"] - 2.0 / 6) < 1e-15
    assert abs(e["rel_l2"] - np.sqrt(2.0) / np.sqrt(27.0)) < 1e-15
    assert abs(e["l1_per_row"] - 2.0 / 3) < 1e-15
    zero = attention.quant_error(o_ref, o_ref)
    assert zero["max_abs"] == 0.0 and zero["rel_l2"] == 0.0


def test_rotation_lowers_the_error_on_outlier_channels():
    """SAW-INT4 page, sections 1-2: naive token-wise INT4 collapses when a few
    channels carry large outliers, and the block-diagonal Hadamard rotation
    spreads them.  The tiny configuration's data (2 channels x20 per head),
    4-bit keys and 2-bit values, quantized with block 64 and with no rotation
    (block 1, the identity)."""
    n, d, hkv = 256, 64, 4
    k = kv_tokens(1001, 0, 1, n, hkv, d, 2, 20.0, 20.0)
    v = kv_tokens(1001, 1, 1, n, hkv, d, 2, 20.0, 20.0)
    q = queries(1001, 0, 1, hkv, d, True)
    pt = page_table(1001, 1, n // 16)
    ref = attention.exact_decode(q, k, v, np.array([n]))
    errs = {}
    for block in (64, 1):
        st = cache.new_state(1, n // 16, d, block, np.array([[[4, 2]] * hkv]))
        cache.append(st, 0, k, v, pt, np.zeros(1, np.int32))
        errs[block] = attention.quant_error(attention.decode(st, 0, q, pt, np.array([n])), ref)
    assert errs[64]["rel_l2"] < errs[1]["rel_l2"]
    assert errs[64]["mean_abs"] < errs[1]["mean_abs"]


def test_keys_with_larger_norms_want_the_bits():
    """"Quantize What Counts: More for Keys, Less for Values": when the keys'
    norms exceed the values', giving the keys the wider codes lowers the
    attention error at the same total bits (K4V2 against K2V4), and K4V2 stays
    within a factor of two of K4V4.
    Keys with 4 outlier channels (x10..50), plain values, as in the
    Llama-3-8B-shaped workload; Hadamard 64."""
    n, d, hkv = 512, 64, 4
    k = kv_tokens(2002, 0, 1, n, hkv, d, 4, 10.0, 50.0)
    v = kv_tokens(2002, 1, 1, n, hkv, d, 0, 1.0, 1.0)
    assert np.linalg.norm(k) > 2 * np.linalg.norm(v)
    q = queries(2002, 0, 1, 4 * hkv, d, True)
    pt = page_table(2002, 1, n // 16)
    ref = attention.exact_decode(q, k, v, np.array([n]))
    err = {}
    for kb, vb in ((4, 2), (2, 4), (4, 4)):
        st = cache.new_state(1, n // 16, d, 64, np.array([[[kb, vb]] * hkv]))
        cache.append(st, 0, k, v, pt, np.zeros(1, np.int32))
        err[(kb, vb)] = attention.quant_error(attention.decode(st, 0, q, pt, np.array([n])),
                                              ref)["rel_l2"]
    # (relative L2 on this data: K4V2 0.53, K2V4 1.04, K4V4 0.31)
    assert err[(4, 2)] < 0.75 * err[(2, 4)], err
    assert err[(4, 4)] < err[(4, 2)] < 2.0 * err[(4, 4)], err

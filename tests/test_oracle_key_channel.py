"""Pins for the oracle's key-per-channel mode: the symmetric per-channel key
quantizer (RateQuant technical summary, Methodology section 3: KIVI's
symmetric per-channel keys; "LogQuant ...", section 5: key-per-channel), its
page layout, the append rule and attention over such a cache."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import attention, cache, layout, quantizer
from workloads import kv_tokens, page_table, queries, round_to_bf16


def _f32(rows):
    return np.asarray(rows, dtype=np.float32)


# ---------------------------------------------------------------- quantizer

def test_worked_example_4bit():
    # Q = 7.  Channel 0: max |u| = 1, fp32(1/7) = 0.142857149..., whose fp16
    # neighbours are 1170/8192 < it < 1171/8192, so s0 = 1171/8192 (rounded up).
    # Channel 1: max |u| = 3, fp32(3/7) = 0.428571432..., fp16 spacing 2^-12
    # there: 1755/4096 < it < 1756/4096, so s1 = 1756/4096 = 439/1024.
    # Codes, round-half-even of u / s:
    #   1 * 8192/1171 = 6.9957 -> 7     -3 * 1024/439 = -6.9977 -> -7
    #   0.5 * 8192/1171 = 3.4979 -> 3    2 * 1024/439 = 4.6651 -> 5
    #   -0.25 * 8192/1171 = -1.7489 -> -2  0 -> 0
    u = _f32([[1.0, -3.0], [0.5, 2.0], [-0.25, 0.0]])
    c, s = quantizer.quantize_channels(u, 4)
    assert [Fraction(float(x)) for x in s] == [Fraction(1171, 8192), Fraction(439, 1024)]
    assert c.tolist() == [[7, -7], [3, 5], [-2, 0]]


def test_worked_example_2bit_three_levels():
    # Q = 1: codes -1, 0, 1.  fp32(0.6) = 0.60000002..., fp16 spacing 2^-11 in
    # [0.5, 1): 1228/2048 < it < 1229/2048, so s = 1229/2048 = 0.60009765625.
    #   0.6 / s = 0.99984 -> 1;  -0.2 / s = -0.33328 -> 0;  0.35 / s = 0.58324 -> 1
    #   -0.6 / s -> -1
    u = _f32([[0.6], [-0.2], [0.35], [-0.6]])
    c, s = quantizer.quantize_channels(u, 2)
    assert Fraction(float(s[0])) == Fraction(1229, 2048)
    assert c[:, 0].tolist() == [1, 0, 1, -1]


def test_ties_round_half_even():
    # max |u| = 0.875 = 7 / 8 -> s = 1/8 exactly; u * 8 = 7, 2.5, 3.5, -2.5, -3.5
    u = _f32([[0.875], [0.3125], [0.4375], [-0.3125], [-0.4375]])
    c, s = quantizer.quantize_channels(u, 4)
    assert float(s[0]) == 0.125
    assert c[:, 0].tolist() == [7, 2, 4, -2, -4]


def _outlier_groups(seed, n_groups=40, d=128):
    rng = np.random.default_rng(seed)
    u = rng.standard_normal((n_groups, 16, d)).astype(np.float32)
    u[:, :, 3] *= 40.0
    u[:, :, 77] *= 0.001
    u[0, :, 5] = 0.0                       # an all-zero channel
    u[1, 3, 9] = 6.0e4                     # near the fp16 limit
    u[2, :, 11] = 1.0e-6                   # subnormal scales
    return u


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_invariants(bits):
    u = _outlier_groups(bits)
    q = quantizer.channel_levels(bits)
    s = quantizer.channel_scales(u, bits)
    raw = quantizer.channel_codes_given(u, s, bits, clip=False)
    assert raw.min() >= -q and raw.max() <= q            # the clamp never fires
    c = quantizer.channel_codes_given(u, s, bits)
    deq = quantizer.dequantize_channels(c, s)
    sf = s.astype(np.float64)[:, None, :]
    assert np.all(np.abs(u - deq) <= sf / 2 * (1 + 1e-6) + 1e-30)
    # the largest |u| of every channel with a normal fp16 scale takes code +-Q
    # (rounding s up costs at most 2^-10 of it); a subnormal scale is coarser
    idx = np.abs(u).argmax(axis=1)
    top = np.take_along_axis(c, idx[:, None, :], axis=1)[:, 0, :]
    normal = s.astype(np.float64) >= 2.0 ** -14
    assert np.all(np.abs(top)[normal] == q)
    assert not normal[2, 11]
    # a zero channel: s = 0 and codes 0
    assert float(s[0, 5]) == 0.0 and not c[0, :, 5].any()
    # symmetric: -u gives the same scales and the negated codes
    c_neg, s_neg = quantizer.quantize_channels(-u, bits)
    assert np.array_equal(s_neg, s) and np.array_equal(c_neg, -c)


def test_eight_bit_grid_is_lossless():
    rng = np.random.default_rng(3)
    e = rng.integers(-6, 6, size=64)
    m = rng.integers(-127, 128, size=(16, 64))
    m[5] = 127                               # every channel reaches +-127
    m[6, ::2] = -127
    u = (m * np.exp2(e)[None, :]).astype(np.float32)
    c, s = quantizer.quantize_channels(u, 8)
    assert np.array_equal(quantizer.dequantize_channels(c, s), u.astype(np.float64))


def test_per_channel_keys_beat_token_wise_on_outlier_channels():
    # KIVI's premise (named on the RateQuant page): key outliers sit in fixed
    # channels, so a scale per channel wastes fewer levels than one per token.
    # Without rotation, at 4 bits, the per-channel key error is the lower one;
    # quantizing along the other axis (a scale per token) is not.
    k = kv_tokens(11, 0, 1, 256, 1, 128, 2, 20.0, 20.0)[0, :, 0].astype(np.float32)
    groups = k.reshape(16, 16, 128)
    c, s = quantizer.quantize_channels(groups, 4)
    mse_channel = np.mean((quantizer.dequantize_channels(c, s) - groups) ** 2)
    ct, st, zt = quantizer.quantize(k, 4)
    mse_token = np.mean((quantizer.dequantize(ct, st, zt) - k) ** 2)
    ct2, st2 = quantizer.quantize_channels(k.reshape(16, 16, 128).transpose(0, 2, 1), 4)
    mse_wrong_axis = np.mean((quantizer.dequantize_channels(ct2, st2).transpose(0, 2, 1)
                              - groups) ** 2)
    assert mse_channel < 0.5 * mse_token
    assert mse_channel < 0.5 * mse_wrong_axis


# ------------------------------------------------------------------- layout

def test_segment_size_and_stored_codes():
    assert layout.head_bytes(128, 4, 4, kpc=True) == 16 * 128 + 256 + 64     # 2368
    assert layout.head_bytes(64, 2, 8, kpc=True) == 16 * (16 + 64) + 128 + 64
    pool = np.zeros((2, layout.page_bytes(64, np.array([[4, 2], [2, 4]]), True)), np.uint8)
    view = layout.PageView(pool, 64, np.array([[4, 2], [2, 4]]), kpc=True)
    codes = np.zeros((16, 64), np.int64)
    codes[0, 0], codes[0, 1] = -7, 7             # offset binary: 1 and 15
    s = np.arange(64).astype(np.float16)
    view.write_key_channels(1, 0, codes, s)
    assert pool[1, 0] == 0xF1                    # element 0 low nibble, element 1 high
    assert pool[1, 2] == 0x88                    # code 0 is stored as 8
    c2, s2 = view.read_key_channels(1, 0)
    assert np.array_equal(c2, codes) and np.array_equal(s2, s)
    # the scales follow the V codes of the same head: 16 * (32 + 16) bytes in
    off = 16 * (64 * 4 // 8 + 64 * 2 // 8)
    assert np.array_equal(pool[1, off:off + 128].view(np.float16), s)


# ------------------------------------------------------------ append rule

def test_quantized_prefix_rule():
    qp = cache.quantized_prefix
    # no window: the full pages; the open page stays in bf16
    assert [qp(n, 0, True) for n in (0, 15, 16, 37, 48)] == [0, 0, 16, 32, 48]
    # window 16: pages that lie wholly before the last 16 positions
    assert [qp(n, 16, True) for n in (16, 31, 32, 37, 63)] == [0, 0, 16, 16, 32]
    # window 5 (not a page multiple)
    assert [qp(n, 5, True) for n in (20, 21, 36, 37)] == [0, 16, 16, 32]
    assert cache.ring_rows(0, True) == 16 and cache.ring_rows(40, True) == 56


def _kpc_state(window, bsz=2, pages=40, d=64, bits=((4, 2), (2, 8)), block=64):
    return cache.new_state(1, pages, d, block, np.array([bits]), window=window,
                           max_batch=bsz, key_per_channel=True)


@pytest.mark.parametrize("window", [0, 5, 16])
def test_chunked_append_equals_single_append(window):
    bsz, d, n = 2, 64, 150
    k = kv_tokens(21, 0, bsz, n, 2, d, 2, 10, 20)
    v = kv_tokens(21, 1, bsz, n, 2, d, 2, 10, 20)
    pt = page_table(21, bsz, 10, 40)
    one = _kpc_state(window)
    cache.append(one, 0, k, v, pt, np.zeros(bsz, np.int32))
    many = _kpc_state(window)
    pos = 0
    for chunk in (1, 14, 1, 16, 3, 33, 40, 42):
        cache.append(many, 0, k[:, pos:pos + chunk], v[:, pos:pos + chunk], pt,
                     np.full(bsz, pos, np.int32))
        pos += chunk
    assert pos == n
    assert np.array_equal(one.pools[0], many.pools[0])
    rows = one.ring_rows
    for p in range(cache.quantized_prefix(n, window, True), n):
        assert np.array_equal(one.windows[0][:, :, :, p % rows],
                              many.windows[0][:, :, :, p % rows])
        assert np.array_equal(one.windows[0][:, :, 0, p % rows], k[:, p])


def test_pages_written_only_when_complete():
    d, bsz = 64, 1
    k = kv_tokens(22, 0, bsz, 40, 2, d, 0, 1, 1)
    v = kv_tokens(22, 1, bsz, 40, 2, d, 0, 1, 1)
    pt = page_table(22, bsz, 4, 8)
    st = _kpc_state(0, bsz=bsz, pages=8)
    cache.append(st, 0, k[:, :15], v[:, :15], pt, np.zeros(bsz, np.int32))
    assert not st.pools[0].any()                     # page 0 still open
    out = cache.append(st, 0, k[:, 15:37], v[:, 15:37], pt, np.full(bsz, 15, np.int32))
    assert out[(0, 0, 0)][0].tolist() == list(range(32))   # pages 0 and 1, not 2
    assert not st.pools[0][pt[0, 2]].any()


def _grid_kv(seed, bsz, n, hkv, d):
    """Keys on a per-channel 8-bit grid (each 16-token page's channels reach
    +-127 steps of a power of two) and values on a per-token 8-bit grid
    (z = -8, s = 1/16, codes 0 and 255 present): both quantize losslessly."""
    rng = np.random.default_rng(seed)
    e = rng.integers(-5, 3, size=(bsz, n // 16, hkv, d))
    m = rng.integers(-127, 128, size=(bsz, n // 16, 16, hkv, d))
    m[:, :, 0] = 127
    k = (m * np.exp2(e)[:, :, None]).reshape(bsz, n, hkv, d).astype(np.float32)
    c = rng.integers(0, 256, size=(bsz, n, hkv, d))
    c[..., 0], c[..., 1] = 0, 255
    v = (c / 16.0 - 8.0).astype(np.float32)
    assert np.array_equal(round_to_bf16(k), k) and np.array_equal(round_to_bf16(v), v)
    return k, v


@pytest.mark.parametrize("window", [0, 7])
def test_lossless_cache_attention_is_exact_attention(window):
    # no rotation, 8-bit codes, inputs on the quantizers' grids: the cache
    # holds K and V exactly, so its attention is plain softmax attention over
    # the inputs (an identity independent of the quantizer's arithmetic)
    bsz, n, hkv, hq, d = 2, 96, 2, 4, 64
    k, v = _grid_kv(31, bsz, n, hkv, d)
    pt = page_table(31, bsz, 8, 16)
    st = _kpc_state(window, bsz=bsz, pages=16, bits=((8, 8), (8, 8)), block=1)
    pos = 0
    for chunk in (17, 1, 30, 48):
        cache.append(st, 0, k[:, pos:pos + chunk], v[:, pos:pos + chunk], pt,
                     np.full(bsz, pos, np.int32))
        pos += chunk
    for length in (n,):
        q = queries(31, 2, bsz, hq, d, True)
        lens = np.full(bsz, length, np.int32)
        got = attention.decode(st, 0, q, pt, lens)
        want = attention.exact_decode(q, k, v, lens)
        assert np.allclose(got, want, rtol=0, atol=1e-12)

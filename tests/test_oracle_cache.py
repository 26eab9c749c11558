"""Pins for oracle.cache: append semantics, window ring, chunking invariance."""
import numpy as np
import pytest

from oracle import cache, hadamard, layout, quantizer
from workloads import kv_tokens, page_table


def _state(window, bsz=2, pages=40, d=64, bits=((4, 2), (8, 4))):
    return cache.new_state(1, pages, d, 32, np.array([bits]), window=window, max_batch=bsz)


@pytest.mark.parametrize("window", [0, 16, 40])
def test_chunked_append_equals_single_append(window):
    bsz, d = 2, 64
    k = kv_tokens(1, 0, bsz, 150, 2, d, 2, 10, 20)
    v = kv_tokens(1, 1, bsz, 150, 2, d, 2, 10, 20)
    pt = page_table(1, bsz, 10, 40)
    one = _state(window)
    cache.append(one, 0, k, v, pt, np.zeros(bsz, np.int32))
    many = _state(window)
    pos = 0
    for chunk in (1, 7, 16, 1, 33, 50, 42):
        cache.append(many, 0, k[:, pos:pos + chunk], v[:, pos:pos + chunk], pt,
                     np.full(bsz, pos, np.int32))
        pos += chunk
    assert pos == 150
    assert np.array_equal(one.pools[0], many.pools[0])
    if window:
        assert np.array_equal(one.windows[0], many.windows[0])


def test_window_holds_the_last_tokens_and_the_rest_is_quantized():
    bsz, d, r, n = 1, 64, 40, 100
    k = kv_tokens(2, 0, bsz, n, 2, d, 0, 1, 1)
    v = kv_tokens(2, 1, bsz, n, 2, d, 0, 1, 1)
    pt = page_table(2, bsz, 10, 40)
    st = _state(r, bsz)
    out = cache.append(st, 0, k, v, pt, np.zeros(bsz, np.int32))
    for p in range(n - r, n):
        assert np.array_equal(st.windows[0][0, :, 0, p % r], k[0, p])
        assert np.array_equal(st.windows[0][0, :, 1, p % r], v[0, p])
    pos, codes, s, z, u32 = out[(0, 1, 0)]
    assert pos.tolist() == list(range(n - r))
    # what was written is the quantization of the rotated input token
    c2, s2, z2 = quantizer.quantize(hadamard.rotate(k[0, :n - r, 1], 32).astype(np.float32), 8)
    assert np.array_equal(codes, c2) and np.array_equal(s, s2) and np.array_equal(z, z2)
    view = st.view(0)
    pages = pt[0, pos // 16]
    rc, rs, rz = view.read(pages, pos % 16, 1, 0)
    assert np.array_equal(rc, c2) and np.array_equal(rs, s2)


def test_untouched_slots_stay_zero():
    st = _state(0, 1)
    k = kv_tokens(3, 0, 1, 5, 2, 64, 0, 1, 1)
    pt = np.arange(10, dtype=np.int32)[None]
    cache.append(st, 0, k, k, pt, np.array([3], np.int32))
    view = st.view(0)
    c, s, z = view.read(np.array([0, 0, 0]), np.array([0, 2, 8]), 0, 0)
    assert not c.any() and not s.astype(np.float64).any()
    c, s, z = view.read(np.array([0]), np.array([3]), 0, 0)
    assert float(s[0]) > 0

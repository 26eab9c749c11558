"""Pins for oracle.logquant: the selection rule's invariants and log spacing,
and attention that reduces to exact bf16 attention when every token is kept."""
import collections
import os

import numpy as np
import pytest

from oracle import attention, cache as ocache, logquant
from tests.conftest import ROOT
from workloads import kv_tokens, page_table, queries


@pytest.mark.parametrize("w", [1, 2, 4, 8, 16])
def test_sizes_order_and_the_kept_ends(w):
    for n in range(0, 24 * w):
        b = logquant.members(n, w)
        assert np.all(np.diff(b) > 0) and (n == 0 or (b[0] >= 0 and b[-1] == n - 1))
        if n < 3 * w:
            assert len(b) == n                      # nothing halved yet
        else:
            assert 2 * w <= len(b) < 3 * w          # the 3W reserve, refilled from 2W
        newest = np.arange(max(0, n - w), n)
        assert np.isin(newest, b).all()             # the newest W tokens are kept
        if n:
            assert b[0] == 0                        # the first of every pair stays


@pytest.mark.parametrize("w", [4, 16, 64])
def test_log_spacing_after_a_halving(w):
    # right after a halving (n = 3W + jW), far enough in: W - 1 gaps of 1, then
    # W / 2 gaps of 2, W / 4 of 4, ..., one of W, and one gap back to position 0
    k = int(np.log2(w))
    n = 3 * w + (k + 4) * w
    b = logquant.members(n, w)
    gaps = collections.Counter(np.diff(b).tolist())
    want = collections.Counter({1: w - 1})
    for j in range(1, k + 1):
        want[2 ** j] += w // 2 ** j
    big = b[1] - b[0]
    gaps[big] -= 1
    assert +gaps == +want and big > w


def _cache(w_bits, n, hkv, d, seed):
    pt = page_table(seed, 1, (n + 15) // 16)
    st = ocache.new_state(1, (n + 15) // 16, d, 64, np.full((1, hkv, 2), w_bits))
    k = kv_tokens(seed, 0, 1, n, hkv, d, 4, 10.0, 50.0)
    v = kv_tokens(seed, 1, 1, n, hkv, d, 4, 10.0, 50.0)
    ocache.append(st, 0, k, v, pt, np.zeros(1, np.int32))
    return st, pt, k, v


def test_every_token_kept_is_exact_attention():
    # n < 3W: B holds every position, so the result is plain bf16 attention
    hkv, d, n, w = 2, 64, 40, 16
    st, pt, k, v = _cache(2, n, hkv, d, 61)
    q = queries(61, 0, 1, 2 * hkv, d, False).astype(np.float64)
    o = logquant.decode(st, 0, q, pt, np.array([n]), w, k, v)
    for h in range(hkv):
        ref = attention.softmax_attention(q[0, 2 * h:2 * h + 2], k[0, :, h], v[0, :, h],
                                          1.0 / np.sqrt(d))
        np.testing.assert_allclose(o[0, 2 * h:2 * h + 2], ref, rtol=0, atol=1e-12)


def test_members_match_the_worked_examples():
    path = os.path.join(ROOT, "tests", "golden", "logquant_members.txt")
    n_cases = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        head, pos = line.split(":")
        w, n = (int(x) for x in head.split())
        assert logquant.members(n, w).tolist() == [int(x) for x in pos.split()], (w, n)
        n_cases += 1
    assert n_cases == 9


def test_lossless_data_gives_the_cached_attention_for_any_window():
    # rotated vectors on the 2-bit grid {-2, -1, 0, 1} (fp16-exact z = -2,
    # s = 1, both ends present) quantize without loss, and x = H u / 64 is
    # bf16-exact: the bf16 rows of B equal the dequantized rows, so the result
    # must equal plain cached attention row for row -- a misplaced row of B
    # (another token's values) would change it
    from oracle.hadamard import unrotate
    rng = np.random.default_rng(63)
    hkv, d, n = 2, 64, 300
    c = rng.integers(0, 4, size=(1, n, hkv, d))
    c[..., 0], c[..., 1] = 0, 3
    u = c.astype(np.float64) - 2.0
    x = unrotate(u, 64)
    assert np.all(x * 64 == np.round(x * 64)) and np.abs(x * 64).max() <= 128
    k, v = x, unrotate(np.flip(u, axis=1).copy(), 64)
    pt = page_table(63, 1, (n + 15) // 16)
    st = ocache.new_state(1, (n + 15) // 16, d, 64, np.full((1, hkv, 2), 2))
    ocache.append(st, 0, k, v, pt, np.zeros(1, np.int32))
    q = queries(63, 0, 1, 2 * hkv, d, False).astype(np.float64)
    plain = attention.decode(st, 0, q, pt, np.array([n]))
    for w in (1, 4, 16, 64):
        np.testing.assert_allclose(logquant.decode(st, 0, q, pt, np.array([n]), w, k, v), plain,
                                   rtol=0, atol=1e-12)

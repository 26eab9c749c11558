"""LogQuant selection in the library (host utility, no GPU) against the oracle.

The library decides membership in B by a closed form of the length (the same
header serves the kernels); the oracle simulates the selection rule of the
LogQuant technical summary, Methodology section 2, token by token."""
import numpy as np
import pytest

import quantized_decode_attention_diag_b300 as kvq
from oracle import logquant


@pytest.mark.parametrize("w", [2, 4, 8, 16, 64, 128])
def test_members_match_the_oracle_selection(w):
    for n in list(range(0, 12 * w)) + [20 * w + 3, 50 * w - 1, 50 * w, 131072]:
        want = logquant.members(n, w)
        got = kvq.kvq_logquant_members(n, w)
        assert np.array_equal(got, want), (w, n)


def test_reserve_sizes():
    assert kvq.kvq_logquant_rows(64) == 3 * 64 + 7 * 32
    assert kvq.kvq_logquant_rows(2) == 6 + 2 * 1
    for bad in (0, 1, 3, 96, 512):
        assert kvq.kvq_logquant_rows(bad) == 0
    with pytest.raises(kvq.KvqError):
        kvq.kvq_logquant_members(10, 48)


def test_descriptor_checks():
    d = kvq.kvq_cache()
    d.num_layers, d.num_kv_heads, d.head_dim, d.page_size = 1, 2, 128, 16
    d.had_block, d.window, d.max_batch, d.num_pages = 128, 0, 3, 10
    bits = np.full((1, 2, 2), 2, np.int8)
    import ctypes
    d.bits_host = bits.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))
    d.logquant_w = 16
    assert kvq.kvq_window_bytes(d) == 3 * 2 * 2 * kvq.kvq_logquant_rows(16) * 128 * 2
    d.window = 32                                  # a window and a reserve: refused
    assert kvq.kvq_window_bytes(d) == 0
    assert "needs window 0" in kvq.kvq_last_error()
    d.window, d.logquant_w = 0, 24                 # not a power of two
    assert kvq.kvq_window_bytes(d) == 0

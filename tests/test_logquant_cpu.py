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


def test_decode_membership_rule_equals_the_host_rule(tmp_path):
    # the decode kernel's masked rounds and member list use 32-bit forms of the
    # closed-form membership and reserve row; compiled from the same header,
    # they must agree with the 64-bit forms that kvq_logquant_members (pinned
    # against the oracle above) uses, for every position of every length up to
    # 12 W and a few long ones
    import os
    import shutil
    import subprocess
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    csrc = os.path.join(os.path.dirname(kvq.LIB_PATH), "csrc")
    src = tmp_path / "lq32.cpp"
    src.write_text(
        '#include <cstdio>\n#include "kvq_logquant.h"\n'
        "int main() {\n"
        "  long long bad = 0, checked = 0;\n"
        "  for (int a = 1; a <= 8; ++a) {\n"
        "    const int w = 1 << a;\n"
        "    const int longs[] = {20 * w + 3, 131072, 131071, 1000003};\n"
        "    for (int n = 0; n < 12 * w + 4; ++n)\n"
        "      for (int p = -1; p <= n; ++p, ++checked)\n"
        "        bad += kvq::lq_member(p, n, w, a) != kvq::lq_member32(p, n, w, a) ||\n"
        "               (p >= 0 && p < n && kvq::lq_member(p, n, w, a) &&\n"
        "                kvq::lq_row(p, n, w, a) != kvq::lq_row32(p, n, w, a));\n"
        "    for (int n : longs)\n"
        "      for (int p = 0; p < n; p += (p < 4 * w || p > n - 16 * w) ? 1 : 7, ++checked)\n"
        "        bad += kvq::lq_member(p, n, w, a) != kvq::lq_member32(p, n, w, a) ||\n"
        "               (kvq::lq_member(p, n, w, a) &&\n"
        "                kvq::lq_row(p, n, w, a) != kvq::lq_row32(p, n, w, a));\n"
        "  }\n"
        '  std::printf("%lld %lld\\n", bad, checked);\n'
        "  return 0;\n}\n")
    exe = tmp_path / "lq32"
    subprocess.run([cxx, "-O1", "-std=c++17", "-I", csrc, str(src), "-o", str(exe)], check=True)
    bad, checked = map(int, subprocess.run([str(exe)], check=True, capture_output=True,
                                           text=True).stdout.split())
    assert checked > 100000 and bad == 0

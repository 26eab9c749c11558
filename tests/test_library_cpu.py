"""C-ABI library on the host: it loads, exports every declared symbol, its
host-only logic (allocator, page geometry, argument checks) matches the oracle.
No call here reaches a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import quantized_decode_attention_diag_b300 as kvq
from oracle import allocator, layout
from tests.conftest import ROOT
from workloads import sensitivities


@pytest.fixture(scope="session", autouse=True)
def built_library():
    from quantized_decode_attention_diag_b300 import build
    build.build()
    return kvq.lib()


def test_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "kvq.h")).read()
    names = sorted(set(re.findall(r"^\s*(?:[\w\*]+\s+)+\**(kvq_\w+)\s*\(", header, re.M)))
    assert {"kvq_append", "kvq_decode_attn", "kvq_alloc_bits", "kvq_page_bytes",
            "kvq_decode_workspace_bytes", "kvq_get_status", "kvq_reset_status",
            "kvq_last_error", "kvq_version"} <= set(names)
    handle = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(handle, n), n
    assert kvq.kvq_version().startswith("kvq")


def _desc(hkv=8, d=128, block=128, bits=(4, 4), layers=1, window=0, pages=64):
    b = np.zeros((layers, hkv, 2), np.int8)
    b[..., 0], b[..., 1] = bits
    desc = kvq.kvq_cache()
    desc.num_layers, desc.num_kv_heads, desc.head_dim, desc.page_size = layers, hkv, d, 16
    desc.had_block, desc.window, desc.max_batch, desc.num_pages = block, window, 4, pages
    desc.bits_host = b.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))
    desc._keep = b
    return desc


@pytest.mark.parametrize("hkv,d,bits", [(8, 128, (4, 4)), (8, 128, (4, 2)), (4, 64, (4, 2)),
                                         (2, 64, (8, 2)), (3, 128, (2, 8))])
def test_page_bytes_matches_layout(hkv, d, bits):
    desc = _desc(hkv=hkv, d=d, block=min(d, 64), bits=bits)
    assert kvq.kvq_page_bytes(desc, 0) == layout.page_bytes(d, np.array([bits] * hkv))


def test_page_bytes_mixed_heads():
    b = np.array([[[4, 2], [8, 4], [4, 4], [2, 2]]], np.int8)
    desc = _desc(hkv=4)
    desc.bits_host = b.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))
    desc._keep = b
    assert kvq.kvq_page_bytes(desc, 0) == layout.page_bytes(128, b[0])


@pytest.mark.parametrize("hkv,d,bits", [(8, 128, (4, 4)), (4, 64, (2, 8)), (3, 128, (8, 2))])
def test_key_per_channel_page_and_ring_bytes(hkv, d, bits):
    desc = _desc(hkv=hkv, d=d, block=min(d, 64), bits=bits, window=5)
    desc.key_per_channel = 1
    assert kvq.kvq_page_bytes(desc, 0) == layout.page_bytes(d, np.array([bits] * hkv), True)
    # a ring of R + 16 rows per (sequence, head, K|V), for max_batch = 4 sequences
    assert kvq.kvq_window_bytes(desc) == 4 * hkv * 2 * (5 + 16) * d * 2
    desc.window = 0
    assert kvq.kvq_window_bytes(desc) == 4 * hkv * 2 * 16 * d * 2


def test_key_per_channel_host_checks():
    fake = 1 << 20
    pools = (ctypes.c_void_p * 1)(fake)
    ap = lambda d: kvq.kvq_append(d, 0, fake, fake, fake, 4, fake, 2, 3, 0)
    desc = _desc()
    desc.layer_pools = pools
    desc.key_per_channel = 1
    assert _checked(ap, desc) == kvq.KVQ_EINVAL         # the ring is needed even with R = 0
    desc.key_per_channel = 2
    assert _checked(ap, desc) == kvq.KVQ_EINVAL
    desc.key_per_channel, desc.logquant_w = 1, 16
    assert _checked(ap, desc) == kvq.KVQ_EUNSUPPORTED   # not built with LogQuant


@pytest.mark.parametrize("seed", range(20))
def test_alloc_bits_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    w = rng.lognormal(0, 1.2, n)
    beta = rng.uniform(3.0, 6.0, n)
    sets = [[2, 4, 8], [4, 8], [2, 4], list(range(1, 9)), [3, 5, 6]]
    allowed = [sets[int(rng.integers(0, len(sets)))] for _ in range(n)]
    lo = sum(min(a) for a in allowed)
    hi = sum(max(a) for a in allowed)
    budget = int(rng.integers(lo, hi + 3))
    want, left = allocator.greedy(w, beta, budget, allowed)
    got, gleft = kvq.kvq_alloc_bits(w, beta, budget, [kvq.mask_of(a) for a in allowed])
    assert got == want and gleft == left


def test_alloc_bits_mixed_layer_config():
    w = sensitivities(1003, 32, 8).reshape(-1)
    allowed = [[4, 8], [2, 4]] * 256
    masks = [kvq.mask_of(a) for a in allowed]
    for budget in (3 * 512, int(3.5 * 512)):
        want, left = allocator.greedy(w, [4.0] * 512, budget, allowed)
        got, gleft = kvq.kvq_alloc_bits(w, [4.0] * 512, budget, masks)
        assert got == want and gleft == left


def test_alloc_bits_errors():
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_alloc_bits([1.0, 1.0], [4.0, 4.0], 5, [kvq.mask_of([4, 8]), kvq.mask_of([2, 4])])
    assert e.value.status == kvq.KVQ_EBUDGET
    for w, beta in (([0.0], [4.0]), ([1.0], [1.0]), ([float("nan")], [4.0])):
        with pytest.raises(kvq.KvqError) as e:
            kvq.kvq_alloc_bits(w, beta, 8)
        assert e.value.status == kvq.KVQ_EINVAL
    bits, left = kvq.kvq_alloc_bits([1.0, 2.0], [4.0, 4.0], 10)   # default {2, 4, 8}
    # (2,2) -> V-like step of the heavier component 2->4, then the other 2->4;
    # no 4->8 step fits the last 2 bits
    assert (bits, left) == ([4, 4], 2)
    assert (bits, left) == tuple(allocator.greedy([1.0, 2.0], [4.0, 4.0], 10, [[2, 4, 8]] * 2))


def _checked(fn, *args):
    with pytest.raises(kvq.KvqError) as e:
        fn(*args)
    return e.value.status


def test_host_argument_checks_run_before_any_device_call():
    fake = 1 << 20                            # never dereferenced: checks fail first
    desc = _desc()
    pools = (ctypes.c_void_p * 1)(fake)
    desc.layer_pools = pools
    ap = lambda d, K=fake, layer=0, B=2, T=3: kvq.kvq_append(d, layer, K, fake, fake, 4, fake,
                                                              B, T, 0)
    assert _checked(ap, desc, 0) == kvq.KVQ_EINVAL              # NULL K
    assert _checked(ap, desc, fake + 8) == kvq.KVQ_EINVAL       # misaligned K
    assert _checked(ap, desc, fake, 1) == kvq.KVQ_EINVAL        # layer out of range
    assert _checked(ap, desc, fake, 0, 0) == kvq.KVQ_EINVAL     # B = 0
    bad = _desc(d=96)
    bad.layer_pools = pools
    assert _checked(ap, bad) == kvq.KVQ_EUNSUPPORTED
    bad = _desc(bits=(3, 4))
    bad.layer_pools = pools
    assert _checked(ap, bad) == kvq.KVQ_EUNSUPPORTED
    bad = _desc(block=16)
    bad.layer_pools = pools
    assert _checked(ap, bad) == kvq.KVQ_EUNSUPPORTED
    nopool = _desc()
    assert _checked(ap, nopool) == kvq.KVQ_EINVAL
    win = _desc(window=16)
    win.layer_pools = pools
    assert _checked(ap, win) == kvq.KVQ_EINVAL                  # window buffer missing
    dec = lambda d, Hq: kvq.kvq_decode_attn(d, 0, fake, 0, fake, 4, fake, 2, Hq, 0.0, fake, fake,
                                             1 << 20, 0)
    assert _checked(dec, desc, 12) == kvq.KVQ_EINVAL            # Hq not a multiple of Hkv
    assert _checked(dec, desc, 64) == kvq.KVQ_EUNSUPPORTED      # GQA group of 8
    assert kvq.kvq_append(desc, 0, fake, fake, fake, 4, fake, 2, 0, 0) is None   # T_new = 0: no-op


# ------------------------------------------------------------ distortion calibration (host)

def test_fit_distortion_matches_the_oracle_fit():
    from oracle import distortion
    rng = np.random.default_rng(21)
    widths = [2, 3, 4, 5, 6]
    b = np.array(widths, np.float64)
    mse = np.stack([rng.uniform(0.1, 3.0) * rng.uniform(3.0, 6.0) ** (-b) *
                    np.exp(rng.normal(0.0, 0.05, size=b.shape)) for _ in range(40)])
    alpha, beta = kvq.kvq_fit_distortion(mse, widths)
    for i in range(40):
        a, bt = distortion.fit(widths, mse[i])
        assert abs(alpha[i] / a - 1) < 1e-10 and abs(beta[i] / bt - 1) < 1e-10


def test_fit_distortion_fallbacks_and_errors():
    alpha, beta = kvq.kvq_fit_distortion([[0.0, 0.0, 2e-3], [0.0, 0.0, 0.0]], [2, 4, 8])
    assert beta.tolist() == [4.0, 4.0]
    assert abs(alpha[0] - 2e-3 * 4.0 ** 8) < 1e-9 and alpha[1] == 0.0
    with pytest.raises(kvq.KvqError):
        kvq.kvq_fit_distortion([[1.0, 0.5]], [4, 4])


def test_distortion_host_checks_run_before_any_device_call():
    fake = 1 << 20                       # never dereferenced: every call fails its checks first
    L = kvq.lib()
    w = np.array([2, 3, 4], np.int32)
    assert L.kvq_distortion(96, 32, 8, fake, 10, w.ctypes.data, 3, fake, 0) == kvq.KVQ_EUNSUPPORTED
    assert L.kvq_distortion(128, 48, 8, fake, 10, w.ctypes.data, 3, fake, 0) == kvq.KVQ_EINVAL
    assert L.kvq_distortion(128, 128, 0, fake, 10, w.ctypes.data, 3, fake, 0) == kvq.KVQ_EINVAL
    assert L.kvq_distortion(128, 128, 8, fake, -1, w.ctypes.data, 3, fake, 0) == kvq.KVQ_EINVAL
    assert L.kvq_distortion(128, 128, 8, fake, 10, w.ctypes.data, 0, fake, 0) == kvq.KVQ_EINVAL
    bad = np.array([2, 9], np.int32)
    assert L.kvq_distortion(128, 128, 8, fake, 10, bad.ctypes.data, 2, fake, 0) == kvq.KVQ_EINVAL
    assert L.kvq_distortion(128, 128, 8, fake + 4, 10, w.ctypes.data, 3, fake, 0) == kvq.KVQ_EINVAL
    assert L.kvq_distortion(128, 128, 8, fake, 10, w.ctypes.data, 3, fake + 4, 0) == kvq.KVQ_EINVAL


def test_descriptor_layout_matches_the_header(tmp_path):
    """The binding's kvq_cache has the C struct's size and field offsets (a C
    program compiled against include/kvq.h prints them)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f for f, _ in kvq.kvq_cache._fields_]
    src = tmp_path / "layout.c"
    src.write_text(
        "#include <stddef.h>\n#include <stdio.h>\n#include \"kvq.h\"\n"
        "int main(void) {\n"
        '  printf("%zu\\n", sizeof(kvq_cache));\n'
        + "".join(f'  printf("%zu\\n", offsetof(kvq_cache, {f}));\n' for f in fields)
        + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert out[0] == ctypes.sizeof(kvq.kvq_cache)
    for f, off in zip(fields, out[1:]):
        assert getattr(kvq.kvq_cache, f).offset == off, f


def test_invariant_divisor_rule(tmp_path):
    # the append kernel divides chunk and row indices by the launch's warps per
    # (head, K|V) group and by T through a multiply-high, an add and a shift;
    # compiled from the same header, that quotient must equal n / d for every
    # divisor up to 4096, powers of two, divisors near 2^31, and dividends at
    # each quotient's edges, near 2^31 and spread between
    import os
    import shutil
    import subprocess
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    cuda_inc = "/usr/local/cuda/include"
    if not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("no CUDA headers")
    root = os.path.dirname(os.path.dirname(kvq.LIB_PATH))
    csrc = os.path.join(os.path.dirname(kvq.LIB_PATH), "csrc")
    src = tmp_path / "fastdiv.cpp"
    src.write_text(
        '#include <cstdio>\n#include <vector>\n#include "kvq_internal.h"\n'
        "int main() {\n"
        "  std::vector<unsigned> ds;\n"
        "  for (unsigned d = 1; d <= 4096; ++d) ds.push_back(d);\n"
        "  for (int k = 13; k <= 30; ++k) { ds.push_back(1u << k); ds.push_back((1u << k) - 1);\n"
        "    ds.push_back((1u << k) + 1); }\n"
        "  for (unsigned d : {2147483647u, 2147483646u, 1073741825u, 16777216u, 131072u, 8192u,\n"
        "                     1000003u, 65537u, 524287u}) ds.push_back(d);\n"
        "  long long bad = 0, checked = 0;\n"
        "  unsigned long long x = 88172645463325252ull;\n"
        "  for (unsigned d : ds) {\n"
        "    const kvq::FastDiv f = kvq::make_fastdiv(d);\n"
        "    auto check = [&](unsigned long long n) {\n"
        "      if (n >= (1ull << 31)) return;\n"
        "      ++checked;\n"
        "      bad += kvq::fastdiv(static_cast<unsigned>(n), f) != n / d;\n"
        "    };\n"
        "    for (unsigned n = 0; n < 3000; ++n) check(n);\n"
        "    for (unsigned long long q = 1; q * d < (1ull << 31); q = q * 3 + 1) {\n"
        "      check(q * d - 1); check(q * d); check(q * d + 1); }\n"
        "    const unsigned long long top = (1ull << 31) - 1;\n"
        "    check(top); check(top - top % d); check(top - top % d - 1);\n"
        "    for (int i = 0; i < 64; ++i) { x ^= x << 13; x ^= x >> 7; x ^= x << 17; check(x % (1ull << 31)); }\n"
        "  }\n"
        '  std::printf("%lld %lld\\n", bad, checked);\n'
        "  return 0;\n}\n")
    exe = tmp_path / "fastdiv"
    subprocess.run([cxx, "-O1", "-std=c++17", "-I", csrc, "-I", os.path.join(root, "include"),
                    "-I", cuda_inc, str(src), "-o", str(exe)], check=True)
    bad, checked = map(int, subprocess.run([str(exe)], check=True, capture_output=True,
                                           text=True).stdout.split())
    assert checked > 10_000_000 and bad == 0

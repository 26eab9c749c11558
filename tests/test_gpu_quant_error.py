"""Quantization error of the whole path against unquantized attention.

For the tiny, the Llama-3-8B-shaped and the long-context configurations, the
GPU quantizes the K/V (kvq_append) with the configuration's Hadamard block and
with no rotation (block 1), decodes, and the oracle measures the error of
attention over the GPU-written cache against attention over the original
bf16 K/V (oracle.attention.exact_decode): max / mean absolute difference,
relative L2 and CriticalKV's L1 output perturbation (CriticalKV technical
summary, Methodology, the perturbation of the attention output).  The GPU's o
is first checked against the oracle over the same cache, so the error
measured is the quantizer's, not the kernel's.  The SAW-INT4 page (sections
1-2) reports that naive token-wise INT4 collapses on outlier channels and
that the block-diagonal rotation repairs it: the rotated cache must have the
lower error.  Errors are printed (``pytest -s``)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quantized_decode_attention_diag_b300 as kvq
from oracle import attention, cache as ocache
from tests.parity import compare_outputs
from tests.test_gpu_parity import _need_gpu  # noqa: F401
from workloads import LLAMA3_8B_LAYER, LONG_CONTEXT, TINY, kv_tokens, page_table, queries


def _dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(torch.bfloat16)


def _dev_i32(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.int32)).cuda()


def _errors(w, pairs, batch=None, ctx=None):
    bsz = batch or w.batch
    n = ctx or w.ctx
    k = kv_tokens(w.seed, 0, bsz, n, w.hkv, w.head_dim, w.k_outliers, w.outlier_lo, w.outlier_hi)
    v = kv_tokens(w.seed, 1, bsz, n, w.hkv, w.head_dim, w.v_outliers, w.outlier_lo, w.outlier_hi)
    q = queries(w.seed, 0, bsz, w.hq, w.head_dim, w.q_fp32)
    mp = n // 16
    pt = page_table(w.seed, bsz, mp)
    lens = np.full(bsz, n, np.int32)
    ref = attention.exact_decode(q, k, v, lens, pairs=pairs)
    kd, vd, ptd = _dev_bf16(k), _dev_bf16(v), _dev_i32(pt)
    qd = torch.from_numpy(q).cuda()
    if not w.q_fp32:
        qd = qd.to(torch.bfloat16)
    bits = np.tile(np.array([w.k_bits, w.v_bits]), (1, w.hkv, 1))
    out = {}
    for block in (w.had_block, 1):
        c = kvq.Cache(1, w.hkv, w.head_dim, block, bits, bsz * mp, window=w.window,
                      max_batch=bsz)
        c.append(0, kd, vd, ptd, _dev_i32(np.zeros(bsz, np.int32)))
        o = c.decode(0, qd, ptd, _dev_i32(lens)).cpu().numpy()
        assert c.get_status() == 0
        st = ocache.CacheState(w.head_dim, block, w.window, bits, [c.pool_host(0)],
                               [c.window_host(0)] if w.window else None)
        o_ora = attention.decode(st, 0, q.astype(np.float64), pt, lens, pairs=pairs)
        compare_outputs(o, o_ora)
        out[block] = {"oracle": attention.quant_error(o_ora, ref),
                      "gpu": attention.quant_error(np.where(np.isnan(ref), np.nan, o), ref)}
        del c
    print(w.name, {b: e["oracle"] for b, e in out.items()})
    return out


def _assert_rotation_helps(out, block):
    for key in ("rel_l2", "mean_abs", "l1_per_row"):
        assert out[block]["oracle"][key] < out[1]["oracle"][key], key


def test_quant_error_tiny():
    out = _errors(TINY, None)
    _assert_rotation_helps(out, TINY.had_block)


def test_quant_error_llama3_8b_layer():
    w = LLAMA3_8B_LAYER
    out = _errors(w, [(0, h) for h in range(w.hkv)] + [(5, 3), (11, 6)])
    _assert_rotation_helps(out, w.had_block)


def test_quant_error_long_context():
    w = LONG_CONTEXT
    out = _errors(w, [(0, 0), (0, 3), (0, 6)])
    _assert_rotation_helps(out, w.had_block)


def test_keys_with_larger_norms_want_the_bits_on_the_gpu():
    """"Quantize What Counts: More for Keys, Less for Values", through the
    kernels: the Llama-3-8B-shaped layer's keys (4 outlier channels x10..50)
    outweigh its values, and at the same total bits the K4V2 cache has the
    lower attention error against unquantized attention than K2V4 (2 sequences
    x 1024 tokens, every head of both)."""
    w = LLAMA3_8B_LAYER
    bsz, n = 2, 1024
    k = kv_tokens(w.seed, 0, bsz, n, w.hkv, w.head_dim, w.k_outliers, w.outlier_lo, w.outlier_hi)
    v = kv_tokens(w.seed, 1, bsz, n, w.hkv, w.head_dim, w.v_outliers, w.outlier_lo, w.outlier_hi)
    assert np.linalg.norm(k) > 2 * np.linalg.norm(v)
    q = queries(w.seed, 0, bsz, w.hq, w.head_dim, False)
    mp = n // 16
    pt = page_table(w.seed, bsz, mp)
    lens = np.full(bsz, n, np.int32)
    ref = attention.exact_decode(q, k, v, lens)
    kd, vd, ptd = _dev_bf16(k), _dev_bf16(v), _dev_i32(pt)
    qd = torch.from_numpy(q).cuda().to(torch.bfloat16)
    err = {}
    for kb, vb in ((4, 2), (2, 4)):
        bits = np.tile(np.array([kb, vb]), (1, w.hkv, 1))
        c = kvq.Cache(1, w.hkv, w.head_dim, w.had_block, bits, bsz * mp, max_batch=bsz)
        c.append(0, kd, vd, ptd, _dev_i32(np.zeros(bsz, np.int32)))
        o = c.decode(0, qd, ptd, _dev_i32(lens)).cpu().numpy()
        assert c.get_status() == 0
        st = ocache.CacheState(w.head_dim, w.had_block, 0, bits, [c.pool_host(0)], None)
        compare_outputs(o, attention.decode(st, 0, q.astype(np.float64), pt, lens))
        err[(kb, vb)] = attention.quant_error(o, ref)["rel_l2"]
    print("relative L2 error", err)
    assert err[(4, 2)] < 0.75 * err[(2, 4)], err

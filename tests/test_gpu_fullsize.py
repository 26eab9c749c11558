"""Full-size workloads on the GPU, checked against the oracle on samples.

* append sweep: 8 sequences x 8192 new tokens, 8 KV heads, head_dim 128, every
  (Hadamard block, bits) pair; block 128 / 4 bits compared on every vector,
  the others on sampled (sequence, head, K|V) groups;
* Llama-3-8B-shaped decode layer: batch 16, 32 q / 8 KV heads, context 4096,
  K4 V4, through the fused decode step the benchmark times (4095 tokens
  prefilled, the 4096th appended by the step); every KV head of sequence 0
  and more sampled pairs under the cluster merge of the full batch, and one
  sequence alone under the ticket merge;
* long context: batch 1, context 131072, K4 V2, 128-token bf16 window; every
  KV head;
* mixed per-head bits: all 32 layers of the batch-64 / context-2048 workload,
  streamed one layer at a time, bits from the RateQuant greedy with (alpha,
  beta) per component calibrated on the GPU (kvq_distortion, kvq_fit_distortion),
  both the stated 3-bit average (K4V2 everywhere) and the 3.5-bit variant.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quantized_decode_attention_diag_b300 as kvq
from oracle import allocator, attention, cache as ocache, quantizer
from tests.parity import compare_outputs, compare_written
from workloads import (APPEND_BITS, APPEND_BLOCKS, APPEND_SWEEP, LLAMA3_8B_LAYER, LONG_CONTEXT,
                       MIXED_32L, kv_tokens, page_table, queries, sensitivities)


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_attention_diag_b300 import build
    build.build()


def dev_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(torch.bfloat16)


def dev_i32(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.int32)).cuda()


def gpu_state(c: kvq.Cache, bits):
    L = c.num_layers
    return ocache.CacheState(c.head_dim, c.had_block, c.window, np.asarray(bits, np.int64),
                             [c.pool_host(l) for l in range(L)],
                             None if not c.window else [c.window_host(l) for l in range(L)])


def _written(k, v, groups, block, bits):
    """Oracle quantization of whole sequences for (b, h, kv) groups (appended at 0)."""
    out = {}
    for (b, h, kv) in groups:
        x = (k if kv == 0 else v)[b, :, h]
        codes, s, z, u32 = quantizer.rotate_and_quantize(x, block, bits[h, kv])
        out[(b, h, kv)] = (np.arange(x.shape[0]), codes, s, z, u32)
    return out


def test_append_sweep_full_size():
    w = APPEND_SWEEP
    bsz, t, hkv, d = w.batch, w.new_tokens, w.hkv, w.head_dim
    k = kv_tokens(w.seed, 0, bsz, t, hkv, d, w.k_outliers, w.outlier_lo, w.outlier_hi)
    v = kv_tokens(w.seed, 1, bsz, t, hkv, d, w.v_outliers, w.outlier_lo, w.outlier_hi)
    kd, vd = dev_bf16(k), dev_bf16(v)
    mp = t // 16
    pt = page_table(w.seed, bsz, mp)
    ptd, lens = dev_i32(pt), dev_i32(np.zeros(bsz, np.int32))
    rng = np.random.default_rng(0)
    total = dict(codes=0, flips=0)
    for block in APPEND_BLOCKS:
        for bits in APPEND_BITS:
            btab = np.full((1, hkv, 2), bits)
            c = kvq.Cache(1, hkv, d, block, btab, bsz * mp)
            c.append(0, kd, vd, ptd, lens)
            torch.cuda.synchronize()
            assert c.get_status() == 0
            if block == 128 and bits == 4:
                groups = [(b, h, kv) for b in range(bsz) for h in range(hkv) for kv in (0, 1)]
            else:
                groups = [(int(rng.integers(bsz)), int(rng.integers(hkv)), kv) for kv in (0, 1)]
            st = compare_written(c.pool_host(0), _written(k, v, groups, block, btab[0]), pt, d,
                                 btab[0])
            total["codes"] += st["codes"]
            total["flips"] += st["flips"]
            del c
    assert total["flips"] < 1e-5 * total["codes"], total


def _prefill(c, layer, k, v, pt, chunk):
    bsz, t = k.shape[:2]
    ptd = dev_i32(pt)
    for t0 in range(0, t, chunk):
        t1 = min(t, t0 + chunk)
        c.append(layer, dev_bf16(k[:, t0:t1]), dev_bf16(v[:, t0:t1]), ptd,
                 dev_i32(np.full(bsz, t0, np.int32)))
    torch.cuda.synchronize()
    assert c.get_status() == 0


def test_decode_llama3_8b_layer_full_size():
    w = LLAMA3_8B_LAYER
    bsz, hkv, d, ctx = w.batch, w.hkv, w.head_dim, w.ctx
    k = kv_tokens(w.seed, 0, bsz, ctx, hkv, d, w.k_outliers, w.outlier_lo, w.outlier_hi)
    v = kv_tokens(w.seed, 1, bsz, ctx, hkv, d, w.v_outliers, w.outlier_lo, w.outlier_hi)
    mp = ctx // 16
    pt = page_table(w.seed, bsz, mp)
    bits = np.full((1, hkv, 2), 4)
    c = kvq.Cache(1, hkv, d, w.had_block, bits, bsz * mp)
    _prefill(c, 0, k[:, :ctx - 1], v[:, :ctx - 1], pt, 1024)
    q = queries(w.seed, 0, bsz, w.hq, d, False)
    lens = np.full(bsz, ctx, np.int32)
    # the benchmark's launch: one fused decode step (token ctx - 1 appended)
    # for the whole batch -- 4 splits per (sequence, KV head), cluster merge
    o = c.decode_step(0, dev_bf16(k[:, ctx - 1]), dev_bf16(v[:, ctx - 1]), dev_bf16(q),
                      dev_i32(pt), dev_i32(lens))
    torch.cuda.synchronize()
    assert c.get_status() == 0
    pairs = [(0, h) for h in range(hkv)] + [(3, 5), (7, 2), (11, 7), (15, 4), (9, 1)]
    st = gpu_state(c, bits)
    ref = attention.decode(st, 0, q.astype(np.float64), pt, lens, pairs=pairs)
    compare_outputs(o.cpu().numpy(), ref)
    # one sequence alone: 32 splits per KV head, ticket merge
    o9 = c.decode(0, dev_bf16(q[9:10]), dev_i32(pt[9:10]), dev_i32(lens[9:10]))
    torch.cuda.synchronize()
    assert c.get_status() == 0
    ref9 = attention.decode(st, 0, q[9:10].astype(np.float64), pt[9:10], lens[9:10],
                            pairs=[(0, h) for h in range(hkv)])
    compare_outputs(o9.cpu().numpy(), ref9)
    assert np.abs(o9.cpu().numpy()[0] - o.cpu().numpy()[9]).max() < 1e-4
    # codes of sampled whole sequences (the step's token included) against the oracle
    compare_written(c.pool_host(0), _written(k, v, [(2, 3, 0), (13, 6, 1), (0, 0, 0)],
                                             w.had_block, bits[0]), pt, d, bits[0])


def test_decode_long_context_full_size():
    w = LONG_CONTEXT
    bsz, hkv, d, ctx, r = w.batch, w.hkv, w.head_dim, w.ctx, w.window
    k = kv_tokens(w.seed, 0, bsz, ctx, hkv, d, w.k_outliers, w.outlier_lo, w.outlier_hi)
    v = kv_tokens(w.seed, 1, bsz, ctx, hkv, d, w.v_outliers, w.outlier_lo, w.outlier_hi)
    mp = ctx // 16
    pt = page_table(w.seed, bsz, mp)
    bits = np.tile(np.array([w.k_bits, w.v_bits]), (1, hkv, 1))
    c = kvq.Cache(1, hkv, d, w.had_block, bits, bsz * mp, window=r, max_batch=bsz)
    _prefill(c, 0, k, v, pt, 16384)
    q = queries(w.seed, 0, bsz, w.hq, d, False)
    lens = np.full(bsz, ctx, np.int32)
    o = c.decode(0, dev_bf16(q), dev_i32(pt), dev_i32(lens))
    torch.cuda.synchronize()
    assert c.get_status() == 0
    st = gpu_state(c, bits)
    ref = attention.decode(st, 0, q.astype(np.float64), pt, lens,
                           pairs=[(0, h) for h in range(hkv)])
    compare_outputs(o.cpu().numpy(), ref)
    # the window holds the last 128 tokens exactly
    for p in (ctx - r, ctx - 1):
        assert np.array_equal(st.windows[0][0, :, 0, p % r], k[0, p])
    # quantized positions cover [0, ctx - r)
    grp = _written(k[:, :ctx - r], v[:, :ctx - r], [(0, 2, 0), (0, 6, 1)], w.had_block, bits[0])
    compare_written(c.pool_host(0), grp, pt, d, bits[0])


def _calibrated_bits(w, avg_bits):
    """Bits [L, Hkv, 2] for the mixed-bits workload: per (layer, K|V) the GPU
    measures each head's quantization MSE at widths 2..6 on a calibration
    sample (2 further sequences x 4096 tokens of the layer's own K/V streams:
    same outlier channels, tokens not in the cache), fits (alpha, beta) per
    component, and the greedy allocates sum(bits) <= avg_bits * 2 L Hkv with
    K in {4, 8} and V in {2, 4} (RateQuant technical summary, Methodology
    sections 1 and 3).  Returns the bits and (alpha, beta)."""
    L, hkv, d = w.num_layers, w.hkv, w.head_dim
    widths = [2, 3, 4, 5, 6]
    mse = np.zeros((L, hkv, 2, len(widths)))
    for l in range(L):
        for kv in range(2):
            x = kv_tokens(w.seed, 2 * l + kv, 2, 4096, hkv, d,
                          w.k_outliers if kv == 0 else w.v_outliers, w.outlier_lo,
                          w.outlier_hi, seq0=w.batch)
            X = dev_bf16(x.reshape(-1, hkv, d))
            mse[l, :, kv] = kvq.kvq_distortion(d, w.had_block, X, widths).cpu().numpy()
    alpha, beta = kvq.kvq_fit_distortion(mse.reshape(-1, len(widths)), widths)
    sens = sensitivities(w.seed, L, hkv).reshape(-1)
    allowed = [[4, 8], [2, 4]] * (L * hkv)
    out = {}
    for avg in avg_bits:
        budget = int(round(avg * L * hkv * 2))
        bits, left = kvq.kvq_alloc_bits(sens * alpha, beta, budget,
                                        [kvq.mask_of(a) for a in allowed])
        want, wleft = allocator.greedy(sens * alpha, beta, budget, allowed)
        assert bits == list(want) and left == wleft
        out[avg] = np.array(bits).reshape(L, hkv, 2)
    return out, alpha, beta


def test_mixed_bits_all_layers_streamed():
    """Every layer of the mixed-bits workload, one at a time (generated,
    appended, decoded, checked, freed): the stated 3-bit average, which the
    greedy can only meet with K4V2 everywhere, and the 3.5-bit variant with
    real K8/V4 upgrades.  Each layer is prefilled with 2047 tokens and takes
    its 2048th through the fused decode step, the launch the benchmark times."""
    w = MIXED_32L
    L, hkv, d, bsz, ctx = w.num_layers, w.hkv, w.head_dim, w.batch, w.ctx
    allocs, alpha, beta = _calibrated_bits(w, (3.0, 3.5))
    assert 3.0 < beta.min() and beta.max() < 6.0   # RateQuant prints 3.6 .. 5.3
    assert np.all(allocs[3.0] == np.array([4, 2]))          # all-minimum allocation
    mixed = allocs[3.5]
    assert len({tuple(x) for x in mixed.reshape(-1, 2)}) > 1
    mp = ctx // 16
    q = queries(w.seed, 0, bsz, w.hq, d, False)
    lens = np.full(bsz, ctx, np.int32)
    rng = np.random.default_rng(1003)
    for layer in range(L):
        k = kv_tokens(w.seed, 2 * layer, bsz, ctx, hkv, d, w.k_outliers, w.outlier_lo,
                      w.outlier_hi)
        v = kv_tokens(w.seed, 2 * layer + 1, bsz, ctx, hkv, d, w.v_outliers, w.outlier_lo,
                      w.outlier_hi)
        kd, vd = dev_bf16(k), dev_bf16(v)
        kpre, vpre = kd[:, :ctx - 1].contiguous(), vd[:, :ctx - 1].contiguous()
        pt = page_table(w.seed, bsz, mp, stream=layer)
        ptd = dev_i32(pt)
        pairs = [(int(rng.integers(bsz)), int(rng.integers(hkv))) for _ in range(2)]
        for avg, bits in allocs.items():
            sub = bits[layer:layer + 1]
            c = kvq.Cache(1, hkv, d, w.had_block, sub, bsz * mp)
            c.append(0, kpre, vpre, ptd, dev_i32(np.zeros(bsz, np.int32)))
            o = c.decode_step(0, kd[:, ctx - 1].contiguous(), vd[:, ctx - 1].contiguous(),
                              dev_bf16(q), ptd, dev_i32(lens))
            torch.cuda.synchronize()
            assert c.get_status() == 0, (layer, avg)
            ref = attention.decode(gpu_state(c, sub), 0, q.astype(np.float64), pt, lens,
                                   pairs=pairs)
            compare_outputs(o.cpu().numpy(), ref)
            b, h = pairs[0]
            compare_written(c.pool_host(0), _written(k, v, [(b, h, 0), (b, h, 1)], w.had_block,
                                                     sub[0]), pt, d, sub[0])
            del c
        del kd, vd, kpre, vpre

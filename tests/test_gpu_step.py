"""kvq_decode_step (one-token append fused into the decode) against the oracle.

The oracle does the plain thing the call stands for: append of the new token
(rotation, quantization, paging, ring) followed by attention over the cache.
Checked after every step: what the GPU wrote for the new (or ring-flushed)
token -- codes and (s, z) by the same rule as the append tests, the bf16 ring
bit for bit -- and o against the oracle's attention over the GPU-written
cache (max-abs 2e-3, mean-abs 2e-4)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quantized_decode_attention_diag_b300 as kvq
from oracle import attention, cache as ocache
from tests.parity import compare_outputs, compare_written
from tests.test_gpu_parity import Pair, dev_bf16, dev_i32, _need_gpu  # noqa: F401
from workloads import kv_tokens, page_table, queries


def _steps(hkv, d, block, bits, lens0, n_steps, window=0, g=4, seed=80):
    """Prefill lens0 tokens with kvq_append, then n_steps fused decode steps."""
    bsz = len(lens0)
    cap = max(lens0) + n_steps
    mp = (cap + 15) // 16 + 1
    pt = page_table(seed, bsz, mp)
    pr = Pair(hkv, d, block, bits, bsz * mp, window=window, max_batch=bsz)
    tot = kv_tokens(seed, 0, bsz, cap, hkv, d, 4, 10.0, 50.0), kv_tokens(seed, 1, bsz, cap, hkv, d,
                                                                          4, 10.0, 50.0)
    # prefill each sequence to its own length (its own window row)
    z1 = np.zeros(1, np.int32)
    for b, l0 in enumerate(lens0):
        if l0:
            kb, vb = tot[0][b:b + 1, :l0], tot[1][b:b + 1, :l0]
            pr.gpu.append(0, dev_bf16(kb), dev_bf16(vb), dev_i32(pt[b:b + 1]), dev_i32(z1),
                          window_row=b)
            written = ocache.append(pr.ora, 0, kb, vb, pt[b:b + 1], z1, window_row=b)
            torch.cuda.synchronize()
            assert pr.gpu.get_status() == 0
            compare_written(pr.gpu.pool_host(0), written, pt[b:b + 1], d, pr.bits[0])
    if window:
        assert np.array_equal(pr.gpu.window_host(0), pr.ora.windows[0])
    ptd = dev_i32(pt)
    lens = np.array(lens0, np.int32)
    worst = dict(max_abs=0.0, mean_abs=0.0)
    for s in range(n_steps):
        kn = np.stack([tot[0][b, lens[b]] for b in range(bsz)])      # [B][Hkv][d]
        vn = np.stack([tot[1][b, lens[b]] for b in range(bsz)])
        q = queries(seed, 10 + s, bsz, hkv * g, d, False)
        qd = torch.from_numpy(q).cuda().to(torch.bfloat16)
        after = lens + 1
        o = pr.gpu.decode_step(0, dev_bf16(kn), dev_bf16(vn), qd, ptd, dev_i32(after))
        torch.cuda.synchronize()
        assert pr.gpu.get_status() == 0
        # the oracle appends the same token, then the GPU-written cache must agree
        written = ocache.append(pr.ora, 0, kn[:, None], vn[:, None], pt, lens)
        compare_written(pr.gpu.pool_host(0), written, pt, d, pr.bits[0])
        if window:
            assert np.array_equal(pr.gpu.window_host(0), pr.ora.windows[0])
        ref = attention.decode(pr.gpu_state(), 0, q.astype(np.float64), pt, after)
        st = compare_outputs(o.cpu().numpy(), ref)
        worst["max_abs"] = max(worst["max_abs"], st["max_abs"])
        worst["mean_abs"] = max(worst["mean_abs"], st["mean_abs"])
        lens = after
    return worst


@pytest.mark.parametrize("lens0", [[0, 15, 16, 31, 300], [4095, 2048]])
def test_step_no_window(lens0):
    _steps(8, 128, 128, (4, 4), lens0, 3)


@pytest.mark.parametrize("bk,bv", [(4, 2), (8, 4), (2, 2)])
def test_step_bit_pairs(bk, bv):
    _steps(4, 128, 64, (bk, bv), [37, 130], 2)


def test_step_head_dim_64_gqa2():
    _steps(2, 64, 32, (4, 2), [1, 64, 100], 2, g=2)


def test_step_mixed_bits_per_head():
    bits = np.array([[[4, 2], [8, 4], [4, 4], [8, 2]]])
    _steps(4, 128, 128, bits, [20, 333], 2)


@pytest.mark.parametrize("lens0", [[0, 5, 126, 127, 128, 129, 400]])
def test_step_with_window(lens0):
    # crosses the window boundary (len <= R: no flush; len > R: the token leaving
    # the ring is quantized into its page) and a page boundary
    _steps(8, 128, 128, (4, 2), lens0, 4, window=128)


def test_step_matches_append_then_decode():
    """The fused call and the two-call sequence give the same cache bytes and o."""
    hkv, d, lens0 = 8, 128, [100, 257]
    bsz = len(lens0)
    mp = 20
    pt = page_table(91, bsz, mp)
    k = kv_tokens(91, 0, bsz, 300, hkv, d, 4, 10.0, 50.0)
    v = kv_tokens(91, 1, bsz, 300, hkv, d, 4, 10.0, 50.0)
    a = Pair(hkv, d, 128, (4, 4), bsz * mp)
    c = Pair(hkv, d, 128, (4, 4), bsz * mp)
    for pr in (a, c):
        for b, l0 in enumerate(lens0):
            pr.gpu.append(0, dev_bf16(k[b:b + 1, :l0]), dev_bf16(v[b:b + 1, :l0]),
                          dev_i32(pt[b:b + 1]), dev_i32(np.zeros(1, np.int32)))
    lens = np.array(lens0, np.int32)
    kn = np.stack([k[b, lens[b]] for b in range(bsz)])
    vn = np.stack([v[b, lens[b]] for b in range(bsz)])
    q = torch.from_numpy(queries(92, 0, bsz, 32, d, False)).cuda().to(torch.bfloat16)
    o1 = a.gpu.decode_step(0, dev_bf16(kn), dev_bf16(vn), q, dev_i32(pt), dev_i32(lens + 1))
    c.gpu.append(0, dev_bf16(kn[:, None]), dev_bf16(vn[:, None]), dev_i32(pt), dev_i32(lens))
    o2 = c.gpu.decode(0, q, dev_i32(pt), dev_i32(lens + 1))
    torch.cuda.synchronize()
    assert np.array_equal(a.gpu.pool_host(0), c.gpu.pool_host(0))
    assert np.abs(o1.cpu().numpy() - o2.cpu().numpy()).max() < 1e-5


def test_step_rejects_a_zero_length():
    pr = Pair(8, 128, 128, (4, 4), 8)
    pt = page_table(93, 1, 4)
    kn = np.zeros((1, 8, 128), np.float32)
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    pr.gpu.decode_step(0, dev_bf16(kn), dev_bf16(kn), q, dev_i32(pt), dev_i32(np.zeros(1, np.int32)))
    torch.cuda.synchronize()

    assert pr.gpu.get_status() & kvq.DEV_BAD_LENGTH
    pr.gpu.reset_status()


@pytest.mark.parametrize("window", [0, 128])
def test_step_overlapped_layers(window):
    """Back-to-back decode steps of several layers launched with programmatic
    dependent launch (each may start while the previous layer's kernel runs),
    eagerly and replayed from a CUDA graph: the same cache bytes and o as
    ordinary launches, and o within tolerance of the oracle."""
    L, hkv, d, g, bsz, t = 4, 8, 128, 4, 3, 700
    mp = t // 16 + 2
    pt = page_table(95, bsz, mp)
    caches = []
    for overlap in (False, True):
        c = kvq.Cache(L, hkv, d, 128, np.full((L, hkv, 2), 4), bsz * mp, window, bsz,
                      overlap=overlap)
        for l in range(L):
            k = kv_tokens(95, 2 * l, bsz, t, hkv, d, 4, 10.0, 50.0)
            v = kv_tokens(95, 2 * l + 1, bsz, t, hkv, d, 4, 10.0, 50.0)
            c.append(l, dev_bf16(k[:, :t - 1]), dev_bf16(v[:, :t - 1]), dev_i32(pt),
                     dev_i32(np.zeros(bsz, np.int32)))
        caches.append((c, k, v))
    torch.cuda.synchronize()
    kn = [dev_bf16(kv_tokens(95, 2 * l, bsz, t, hkv, d, 4, 10.0, 50.0)[:, t - 1]) for l in range(L)]
    vn = [dev_bf16(kv_tokens(95, 2 * l + 1, bsz, t, hkv, d, 4, 10.0, 50.0)[:, t - 1])
          for l in range(L)]
    q = [torch.from_numpy(queries(96, l, bsz, hkv * g, d, False)).cuda().to(torch.bfloat16)
         for l in range(L)]
    ptd, lens = dev_i32(pt), dev_i32(np.full(bsz, t, np.int32))
    outs = []
    for c, _, _ in caches:
        o = torch.zeros((L, bsz, hkv * g, d), dtype=torch.float32, device="cuda")
        ws = c.workspace(bsz, hkv * g, mp)
        for l in range(L):
            c.decode_step(l, kn[l], vn[l], q[l], ptd, lens, o=o[l], workspace=ws)
        torch.cuda.synchronize()
        assert c.get_status() == 0
        first = o.clone()
        if window:   # a step moves the ring: repeating it is not idempotent
            outs.append(o.cpu().numpy())
            continue
        # the same steps from a graph (the step re-appends the same token: idempotent)
        o.zero_()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=s):
                for l in range(L):
                    c.decode_step(l, kn[l], vn[l], q[l], ptd, lens, o=o[l], workspace=ws)
            for _ in range(3):
                gr.replay()
        torch.cuda.synchronize()
        assert c.get_status() == 0
        assert torch.equal(first, o)
        outs.append(o.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    for l in range(L):
        assert np.array_equal(caches[0][0].pool_host(l), caches[1][0].pool_host(l))
        if window:
            assert np.array_equal(caches[0][0].window_host(l), caches[1][0].window_host(l))
    c = caches[1][0]
    for l in (0, L - 1):
        st = ocache.CacheState(d, 128, window, c.bits, [c.pool_host(x) for x in range(L)],
                               None if not window else [c.window_host(x) for x in range(L)])
        ref = attention.decode(st, l, queries(96, l, bsz, hkv * g, d, False).astype(np.float64),
                               pt, np.full(bsz, t, np.int32))
        compare_outputs(outs[1][l], ref)


@pytest.mark.parametrize("window", [0, 64])
def test_step_mixed_segment_sizes(window):
    # 8-bit keys beside 2- and 4-bit ones: the largest page segment sets the
    # layer's stage size, the narrower heads' copies fill part of a stage; a
    # short sequence (cluster merge) and a long one (ticket merge)
    bits = np.array([[[4, 2], [8, 4], [8, 4], [4, 4], [2, 2], [8, 8], [4, 2], [4, 2]]])
    _steps(8, 128, 128, bits, [40, 3000], 20, window=window)


def test_step_ticket_merge_for_wide_segments():
    # 8-bit keys with 4-bit values (3200-byte stages) beside 4-bit keys, 18
    # sequences x 8 KV heads: four CTAs per SM give 4 splits per unit on 148
    # SMs, and a cluster merge's receive buffer for 4 partials would leave 3
    # CTAs per SM, so the splits merge through global memory instead
    bits = np.array([[[8, 4], [4, 2]] * 4])
    _steps(8, 128, 128, bits, [520] * 18, 2)

"""CUDA path vs the CPU oracle, element by element, on seeded inputs.

Every test calls the C-ABI library through its Python binding; the oracle runs
on the same inputs (and, for attention, over the cache the GPU wrote)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quantized_decode_attention_diag_b300 as kvq
from oracle import attention, cache as ocache
from tests.parity import compare_outputs, compare_written
from workloads import kv_tokens, page_table, queries, ragged_lengths


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


class Pair:
    """A GPU cache and the oracle's cache driven through the same appends."""

    def __init__(self, hkv, d, block, bits, num_pages, window=0, max_batch=4, layers=1):
        bits = np.broadcast_to(np.asarray(bits, np.int64), (layers, hkv, 2)).copy()
        self.bits = bits
        self.d = d
        self.gpu = kvq.Cache(layers, hkv, d, block, bits, num_pages, window, max_batch)
        self.ora = ocache.new_state(layers, num_pages, d, block, bits, window, max_batch)

    def append(self, layer, k, v, pt, lens_before):
        self.gpu.append(layer, dev_bf16(k), dev_bf16(v), dev_i32(pt), dev_i32(lens_before))
        written = ocache.append(self.ora, layer, k, v, pt, lens_before)
        torch.cuda.synchronize()
        assert self.gpu.get_status() == 0
        stats = compare_written(self.gpu.pool_host(layer), written, pt, self.d, self.bits[layer])
        if self.ora.windows is not None:
            assert np.array_equal(self.gpu.window_host(layer), self.ora.windows[layer])
        return stats

    def gpu_state(self):
        st = ocache.CacheState(self.d, self.ora.had_block, self.ora.window, self.bits,
                               [self.gpu.pool_host(l) for l in range(self.bits.shape[0])],
                               None if not self.ora.window else
                               [self.gpu.window_host(l) for l in range(self.bits.shape[0])])
        return st

    def decode_check(self, layer, q, pt, lens, q_fp32=False, pairs=None):
        qd = torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda()
        if not q_fp32:
            qd = qd.to(torch.bfloat16)      # q holds bf16-exact values
        o = self.gpu.decode(layer, qd, dev_i32(pt), dev_i32(lens))
        torch.cuda.synchronize()
        assert self.gpu.get_status() == 0
        ref = attention.decode(self.gpu_state(), layer, q.astype(np.float64), pt, lens, pairs=pairs)
        return compare_outputs(o.cpu().numpy(), ref)


def _kv(seed, b, t, hkv, d, outl=4, lo=10.0, hi=50.0, start=0):
    return (kv_tokens(seed, 0, b, t, hkv, d, outl, lo, hi, start),
            kv_tokens(seed, 1, b, t, hkv, d, outl, lo, hi, start))


# ------------------------------------------------------------------------ append parity

@pytest.mark.parametrize("block", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_append_blocks_and_bits(block, bits):
    hkv, d, bsz, t = 2, 128, 2, 100
    pt = page_table(7, bsz, 8)
    pr = Pair(hkv, d, block, (bits, bits), bsz * 8)
    k, v = _kv(20 + block + bits, bsz, t, hkv, d)
    stats = pr.append(0, k, v, pt, np.array([0, 7], np.int32))
    assert stats["vectors"] == bsz * t * hkv * 2


@pytest.mark.parametrize("block", [32, 64])
@pytest.mark.parametrize("bits", [(4, 2), (8, 2), (2, 8), (8, 4)])
def test_append_head_dim_64(block, bits):
    pt = page_table(8, 1, 20)
    pr = Pair(4, 64, block, bits, 20)
    k, v = _kv(30, 1, 256, 4, 64, outl=2, lo=20.0, hi=20.0)
    pr.append(0, k, v, pt, np.array([0], np.int32))


def test_append_mixed_bits_per_head():
    bits = np.array([[[4, 2], [8, 4], [2, 2], [4, 8]]])
    pt = page_table(9, 3, 6)
    pr = Pair(4, 128, 128, bits, 18)
    k, v = _kv(31, 3, 37, 4, 128)
    pr.append(0, k, v, pt, np.array([3, 0, 50], np.int32))


def test_append_single_tokens_then_chunks():
    pt = page_table(10, 5, 6)
    pr = Pair(8, 128, 128, (4, 4), 30)
    lens = np.array([0, 15, 16, 17, 31], np.int32)
    for step, t in enumerate((1, 1, 3, 16, 1, 20)):
        k, v = _kv(40 + step, 5, t, 8, 128)
        pr.append(0, k, v, pt, lens)
        lens = lens + t


@pytest.mark.parametrize("window", [16, 40, 128])
def test_append_with_window(window):
    bsz = 3
    pt = page_table(11, bsz, 20)
    pr = Pair(2, 128, 64, (4, 2), bsz * 20, window=window, max_batch=bsz)
    lens = np.array([0, 5, 33], np.int32)
    for step, t in enumerate((30, 1, 1, 16, 50, 1, 130, 2)):
        k, v = _kv(50 + step, bsz, t, 2, 128)
        pr.append(0, k, v, pt, lens)
        lens = lens + t


# ------------------------------------------------------------------------ decode parity

def _filled_pair(hkv, d, block, bits, lens, window=0, seed=60, max_pages=None, outl=4):
    bsz = len(lens)
    mp = max_pages or max(1, (max(lens) + 15) // 16)
    pt = page_table(seed, bsz, mp)
    pr = Pair(hkv, d, block, bits, bsz * mp, window=window, max_batch=bsz)
    k, v = _kv(seed, bsz, max(lens), hkv, d, outl=outl)
    # a ragged batch: each sequence is appended with its own length
    for b in range(bsz):
        if lens[b]:
            pr.gpu.append(0, dev_bf16(k[b:b + 1, :lens[b]]), dev_bf16(v[b:b + 1, :lens[b]]),
                          dev_i32(pt[b:b + 1]), dev_i32(np.zeros(1, np.int32)))
    torch.cuda.synchronize()
    assert pr.gpu.get_status() == 0
    return pr, pt, k, v


def test_decode_tiny_fp32_query():
    # 1 layer, batch 1, 4 q heads = 4 KV heads, head_dim 64, context 256, K4 V2, block 64
    pr, pt, k, v = _filled_pair(4, 64, 64, (4, 2), [256], outl=2)
    q = queries(1001, 0, 1, 4, 64, True)
    pr.decode_check(0, q, pt, np.array([256], np.int32), q_fp32=True)


@pytest.mark.parametrize("window", [0, 128])
def test_decode_split_limit_ticket_merge(window):
    # one sequence, one KV head (4 query heads), 65536 tokens: the wave leaves
    # this unit all 592 slots, so it takes the split limit, 256 splits of 16
    # pages (257 CTAs with the window), merged through global memory by the
    # last CTA -- the combine's largest partial count
    pr, pt, k, v = _filled_pair(1, 128, 128, (4, 2), [65536], window=window)
    q = queries(1003, 0, 1, 4, 128, False)
    pr.decode_check(0, q, pt, np.array([65536], np.int32))


@pytest.mark.parametrize("lens", [[1, 300, 77], [4096, 4000], [16, 17, 15, 0]])
def test_decode_gqa4_ragged(lens):
    pr, pt, k, v = _filled_pair(8, 128, 128, (4, 4), lens)
    q = queries(62, 0, len(lens), 32, 128, False)
    pr.decode_check(0, q, pt, np.array(lens, np.int32))


def test_decode_split_count_invariance():
    lens = [700, 333]
    pr, pt, k, v = _filled_pair(8, 128, 128, (4, 2), lens)
    q = queries(63, 0, 2, 32, 128, False)
    outs = []
    for mp in (pt.shape[1], pt.shape[1] * 3, pt.shape[1] * 9):
        ptd = np.pad(pt, ((0, 0), (0, mp - pt.shape[1])), constant_values=-1)
        o = pr.gpu.decode(0, torch.from_numpy(q).cuda().to(torch.bfloat16), dev_i32(ptd),
                          dev_i32(np.array(lens, np.int32)))
        outs.append(o.cpu().numpy())
    assert np.abs(outs[0] - outs[1]).max() < 1e-4 and np.abs(outs[0] - outs[2]).max() < 1e-4
    pr.decode_check(0, q, pt, np.array(lens, np.int32))


@pytest.mark.parametrize("bk", [2, 4, 8])
@pytest.mark.parametrize("bv", [2, 4, 8])
def test_decode_all_bit_pairs_head_dim_64(bk, bv):
    pr, pt, k, v = _filled_pair(2, 64, 32, (bk, bv), [130, 61])
    q = queries(64, 0, 2, 4, 64, False)
    pr.decode_check(0, q, pt, np.array([130, 61], np.int32))


@pytest.mark.parametrize("bk,bv", [(8, 8), (2, 2), (8, 2)])
def test_decode_bit_pairs_head_dim_128(bk, bv):
    pr, pt, k, v = _filled_pair(4, 128, 128, (bk, bv), [515, 64])
    q = queries(65, 0, 2, 16, 128, False)
    pr.decode_check(0, q, pt, np.array([515, 64], np.int32))


def test_decode_mixed_bits_and_gqa2():
    bits = np.array([[[4, 2], [8, 4], [4, 4], [8, 2]]])
    pr, pt, k, v = _filled_pair(4, 128, 128, bits, [200, 333])
    q = queries(66, 0, 2, 8, 128, False)
    pr.decode_check(0, q, pt, np.array([200, 333], np.int32))


@pytest.mark.parametrize("lens", [[5, 127, 128, 129, 500]])
def test_decode_with_window(lens):
    pr, pt, k, v = _filled_pair(8, 128, 128, (4, 2), lens, window=128)
    q = queries(67, 0, len(lens), 32, 128, False)
    pr.decode_check(0, q, pt, np.array(lens, np.int32))


def test_decode_empty_and_single_token():
    pr, pt, k, v = _filled_pair(8, 128, 128, (4, 4), [0, 1, 2])
    q = queries(68, 0, 3, 32, 128, False)
    st = pr.decode_check(0, q, pt, np.array([0, 1, 2], np.int32))
    assert st["n"] > 0


# ------------------------------------------------------------------------ device errors

def test_bad_page_id_sets_status_and_skips():
    pr, pt, k, v = _filled_pair(8, 128, 128, (4, 4), [64])
    bad = pt.copy()
    bad[0, 1] = 10 ** 6
    q = torch.from_numpy(queries(69, 0, 1, 32, 128, False)).cuda().to(torch.bfloat16)
    pr.gpu.decode(0, q, dev_i32(bad), dev_i32(np.array([64], np.int32)))
    torch.cuda.synchronize()
    assert pr.gpu.get_status() & kvq.DEV_BAD_PAGE
    pr.gpu.reset_status()
    kk, vv = _kv(70, 1, 20, 8, 128)
    pr.gpu.append(0, dev_bf16(kk), dev_bf16(vv), dev_i32(bad), dev_i32(np.array([16], np.int32)))
    torch.cuda.synchronize()
    assert pr.gpu.get_status() & kvq.DEV_BAD_PAGE
    pr.gpu.reset_status()
    pr.gpu.decode(0, q, dev_i32(pt), dev_i32(np.array([10 ** 5], np.int32)))
    torch.cuda.synchronize()
    assert pr.gpu.get_status() & kvq.DEV_BAD_LENGTH
    pr.gpu.reset_status()
    torch.cuda.synchronize()
    assert pr.gpu.get_status() == 0


# ------------------------------------------------------- running maximum of the softmax

def test_decode_rising_scores():
    """Scores that climb across the sequence: the running maximum is raised in
    many steps and lags the scores in between (p > 1 within the slack)."""
    hkv, d, g, bsz, t = 2, 128, 4, 2, 700
    pr = Pair(hkv, d, 128, (4, 4), bsz * 48, max_batch=bsz)
    pt = page_table(131, bsz, 48)
    k, v = _kv(131, bsz, t, hkv, d, outl=0)
    ramp = 1.8 * np.arange(t, dtype=np.float32) / t
    k = k + ramp[None, :, None, None]
    k = torch.from_numpy(k).to(torch.bfloat16).float().numpy()    # bf16-exact
    pr.append(0, k, v, pt, np.zeros(bsz, np.int32))
    q = queries(131, 0, bsz, hkv * g, d, False) + 2.0
    q = torch.from_numpy(q).to(torch.bfloat16).float().numpy()
    pr.decode_check(0, q, pt, np.array([t, t - 5], np.int32))


def test_decode_large_value_scales():
    """Values scaled by 2^9: p s leaves the fp16 range under a lagging running
    maximum, so those rounds take the exact maximum.  o scales exactly."""
    hkv, d, g, bsz, t = 2, 128, 4, 2, 600
    pr = Pair(hkv, d, 128, (4, 4), bsz * 40, max_batch=bsz)
    pt = page_table(132, bsz, 40)
    k, v = _kv(132, bsz, t, hkv, d, outl=0)
    ramp = 1.8 * np.arange(t, dtype=np.float32) / t
    k = torch.from_numpy(k + ramp[None, :, None, None]).to(torch.bfloat16).float().numpy()
    v = v * 512.0
    pr.gpu.append(0, dev_bf16(k), dev_bf16(v), dev_i32(pt), dev_i32(np.zeros(bsz, np.int32)))
    torch.cuda.synchronize()
    assert pr.gpu.get_status() == 0
    q = queries(132, 0, bsz, hkv * g, d, False) + 2.0
    q = torch.from_numpy(q).to(torch.bfloat16).float().numpy()
    lens = np.array([t, t - 7], np.int32)
    o = pr.gpu.decode(0, torch.from_numpy(q).cuda().to(torch.bfloat16), dev_i32(pt), dev_i32(lens))
    torch.cuda.synchronize()
    assert pr.gpu.get_status() == 0
    ref = attention.decode(pr.gpu_state(), 0, q.astype(np.float64), pt, lens)
    compare_outputs(o.cpu().numpy() / 512.0, ref / 512.0)


def test_decode_overlapped_layers_match_ordinary_launches():
    """kvq_decode_attn over several layers back to back with
    KVQ_LAUNCH_OVERLAP (programmatic dependent launch): the same o, bit for
    bit, as ordinary launches, and within tolerance of the oracle."""
    # 16 sequences x 8 KV heads: 128 units, 4 splits each, merged in clusters;
    # the static-entry test covers the ticket merge under overlap
    L, hkv, d, g, bsz, t = 3, 8, 128, 4, 16, 900
    mp = t // 16 + 1
    pt = page_table(97, bsz, mp)
    lens = np.array([t, 450, 17, 1, 899, 640, 333, 16] * 2, np.int32)
    outs = []
    for overlap in (False, True):
        c = kvq.Cache(L, hkv, d, 64, np.full((L, hkv, 2), 4), bsz * mp, overlap=overlap)
        for l in range(L):
            k = kv_tokens(97, 2 * l, bsz, t, hkv, d, 4, 10.0, 50.0)
            v = kv_tokens(97, 2 * l + 1, bsz, t, hkv, d, 4, 10.0, 50.0)
            c.append(l, dev_bf16(k), dev_bf16(v), dev_i32(pt), dev_i32(np.zeros(bsz, np.int32)))
        torch.cuda.synchronize()
        qs = [queries(98, l, bsz, hkv * g, d, False) for l in range(L)]
        ptd, lensd = dev_i32(pt), dev_i32(lens)
        o = [c.decode(l, torch.from_numpy(qs[l]).cuda().to(torch.bfloat16), ptd, lensd)
             for l in range(L)]
        torch.cuda.synchronize()
        assert c.get_status() == 0
        outs.append([x.cpu().numpy() for x in o])
        if overlap:
            for l in (0, L - 1):
                st = ocache.CacheState(d, 64, 0, c.bits, [c.pool_host(x) for x in range(L)], None)
                ref = attention.decode(st, l, qs[l].astype(np.float64), pt, lens)
                compare_outputs(outs[1][l], ref)
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_tiny_exact_config():
    """The tiny correctness configuration exactly as stated: 1 layer, batch 1,
    4 q = 4 KV heads, head_dim 64, context 256, fp32 q, K and V ~ N(0, 1) with 2
    seeded outlier channels per head scaled x20, Hadamard block 64, K INT4 /
    V INT2, page 16.  Codes and (s, z) end to end against the oracle's own
    append of the same inputs; o against the oracle over the GPU-written cache."""
    from workloads import TINY as w
    k = kv_tokens(w.seed, 0, 1, w.ctx, w.hkv, w.head_dim, w.k_outliers, w.outlier_lo,
                  w.outlier_hi)
    v = kv_tokens(w.seed, 1, 1, w.ctx, w.hkv, w.head_dim, w.v_outliers, w.outlier_lo,
                  w.outlier_hi)
    assert w.outlier_lo == w.outlier_hi == 20.0 and w.k_outliers == w.v_outliers == 2
    pt = page_table(w.seed, 1, w.ctx // 16)
    pr = Pair(w.hkv, w.head_dim, w.had_block, (w.k_bits, w.v_bits), w.ctx // 16)
    stats = pr.append(0, k, v, pt, np.zeros(1, np.int32))
    assert stats["vectors"] == w.ctx * w.hkv * 2
    q = queries(w.seed, 0, 1, w.hq, w.head_dim, True)
    pr.decode_check(0, q, pt, np.array([w.ctx], np.int32), q_fp32=True)


@pytest.mark.parametrize("bits", [(4, 2), (8, 4)])
def test_no_rotation_block_1(bits):
    """Hadamard block 1 (no rotation, u = x): append and decode against the
    oracle, whose block-1 'rotation' is the identity matrix."""
    pr, pt, k, v = _filled_pair(4, 128, 1, bits, [300, 45])
    q = queries(68, 0, 2, 16, 128, False)
    pr.decode_check(0, q, pt, np.array([300, 45], np.int32))
    pr2 = Pair(4, 128, 1, bits, 40)
    pt2 = page_table(69, 2, 20)
    kk, vv = _kv(69, 2, 70, 4, 128)
    pr2.append(0, kk, vv, pt2, np.array([0, 3], np.int32))

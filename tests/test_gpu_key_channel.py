"""Key-per-channel mode on the GPU against the oracle.

Keys are quantized symmetrically per channel over each page (one fp16 scale
per page, KV head and channel), values token-wise; a page is quantized once all
of its positions have left the window, and the rest waits in a bf16 ring of
R + 16 rows (RateQuant technical summary, Methodology section 3: KIVI's
symmetric per-channel keys and asymmetric per-token values; "LogQuant ...",
section 5: key-per-channel).  Checked: the channel scales and codes the append
writes, the ring, decode attention over the GPU-written cache (cluster and
ticket merges, every GQA group, both query types, with and without rotation),
and the decode step (the append of its token, then the decode)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quantized_decode_attention_diag_b300 as kvq
from oracle import attention, cache as ocache
from tests.parity import compare_key_channels, compare_outputs, compare_written
from tests.test_gpu_parity import _need_gpu, dev_bf16, dev_i32  # noqa: F401
from workloads import kv_tokens, page_table, queries


class KpcPair:
    """A key-per-channel GPU cache and the oracle's, driven through the same appends."""

    def __init__(self, hkv, d, block, bits, num_pages, window=0, max_batch=4):
        self.bits = np.broadcast_to(np.asarray(bits, np.int64), (1, hkv, 2)).copy()
        self.d, self.block, self.window = d, block, window
        self.gpu = kvq.Cache(1, hkv, d, block, self.bits, num_pages, window, max_batch,
                             key_per_channel=True)
        self.ora = ocache.new_state(1, num_pages, d, block, self.bits, window, max_batch,
                                    key_per_channel=True)

    def check_written(self, written, pt):
        pool = self.gpu.pool_host(0)
        a = compare_key_channels(pool, written, pt, self.d, self.bits[0])
        b = compare_written(pool, written, pt, self.d, self.bits[0], kpc=True)
        assert np.array_equal(self.gpu.window_host(0), self.ora.windows[0])
        return a, b

    def append(self, k, v, pt, lens_before):
        self.gpu.append(0, dev_bf16(k), dev_bf16(v), dev_i32(pt), dev_i32(lens_before))
        written = ocache.append(self.ora, 0, k, v, pt, lens_before)
        torch.cuda.synchronize()
        assert self.gpu.get_status() == 0
        return self.check_written(written, pt)

    def gpu_state(self):
        return ocache.CacheState(self.d, self.block, self.window, self.bits,
                                 [self.gpu.pool_host(0)], [self.gpu.window_host(0)], True)

    def decode_check(self, q, pt, lens, q_fp32=False, pairs=None):
        qd = torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda()
        if not q_fp32:
            qd = qd.to(torch.bfloat16)
        o = self.gpu.decode(0, qd, dev_i32(pt), dev_i32(lens))
        torch.cuda.synchronize()
        assert self.gpu.get_status() == 0
        ref = attention.decode(self.gpu_state(), 0, q.astype(np.float64), pt, lens, pairs=pairs)
        return compare_outputs(o.cpu().numpy(), ref)


def _kv(seed, b, t, hkv, d, start=0):
    return (kv_tokens(seed, 0, b, t, hkv, d, 4, 10.0, 50.0, start),
            kv_tokens(seed, 1, b, t, hkv, d, 4, 10.0, 50.0, start))


@pytest.mark.parametrize("d,block,bits,window", [
    (128, 128, (4, 4), 0), (128, 1, (2, 2), 0), (128, 64, (8, 4), 24), (64, 64, (4, 2), 5),
    (64, 1, (2, 8), 16), (128, 32, (4, 2), 40)])
def test_chunked_appends_then_decode(d, block, bits, window):
    bsz, hkv, g = 3, 2, 4
    mp = 24
    pt = page_table(300 + d + window, bsz, mp)
    pair = KpcPair(hkv, d, block, bits, bsz * mp, window, max_batch=bsz)
    k, v = _kv(300 + window, bsz, 300, hkv, d)
    pos = 0
    for chunk in (37, 1, 15, 16, 2, 64, 1, 100, 33, 31):
        pair.append(k[:, pos:pos + chunk], v[:, pos:pos + chunk], pt, np.full(bsz, pos, np.int32))
        pos += chunk
        if chunk in (15, 64, 31):
            q = queries(301 + pos, 0, bsz, g * hkv, d, False)
            pair.decode_check(q, pt, np.full(bsz, pos, np.int32))
    assert pos == 300


@pytest.mark.parametrize("g,q_fp32", [(1, True), (2, False), (4, True)])
@pytest.mark.parametrize("ctx", [200, 5000])          # cluster merge / ticket merge
def test_decode_groups_and_merges(g, q_fp32, ctx):
    bsz, hkv, d = 2, 4, 128
    mp = (ctx + 15) // 16
    pt = page_table(310 + ctx, bsz, mp)
    pair = KpcPair(hkv, d, 128, (4, 2), bsz * mp, 0, max_batch=bsz)
    k, v = _kv(311, bsz, ctx, hkv, d)
    pair.append(k, v, pt, np.zeros(bsz, np.int32))
    lens = np.array([ctx, ctx - 7], np.int32)
    q = queries(312 + g, 0, bsz, g * hkv, d, q_fp32)
    pair.decode_check(q, pt, lens, q_fp32)


@pytest.mark.parametrize("d,g,bits", [(128, 4, (4, 2)), (64, 2, (4, 2)), (128, 4, (2, 2)),
                                      (64, 1, (2, 4))])
def test_open_page_in_the_last_split(d, g, bits):
    # without a window the open page's bf16 rows (at most 15) are attended by
    # the last quantized split itself: lengths around page boundaries, and
    # sequences with no full page at all
    lens = np.array([1, 7, 15, 16, 17, 40, 47, 300], np.int32)
    bsz, hkv = len(lens), 2
    mp = 20
    pt = page_table(340 + d, bsz, mp)
    pair = KpcPair(hkv, d, d, bits, bsz * mp, 0, max_batch=bsz)
    k, v = _kv(341, bsz, int(lens.max()), hkv, d)
    for b in range(bsz):
        pair.gpu.append(0, dev_bf16(k[b:b + 1, :lens[b]]), dev_bf16(v[b:b + 1, :lens[b]]),
                        dev_i32(pt[b:b + 1]), dev_i32(np.zeros(1, np.int32)), window_row=b)
        ocache.append(pair.ora, 0, k[b:b + 1, :lens[b]], v[b:b + 1, :lens[b]], pt[b:b + 1],
                      np.zeros(1, np.int32), window_row=b)
    torch.cuda.synchronize()
    assert pair.gpu.get_status() == 0
    assert np.array_equal(pair.gpu.window_host(0), pair.ora.windows[0])
    for q_fp32 in (False, True):
        q = queries(342 + d, int(q_fp32), bsz, g * hkv, d, q_fp32)
        pair.decode_check(q, pt, lens, q_fp32)


def test_ragged_prefills_one_sequence_at_a_time():
    bsz, hkv, d, window = 4, 2, 128, 20
    lens = np.array([0, 9, 16, 333], np.int32)
    mp = 24
    pt = page_table(320, bsz, mp)
    pair = KpcPair(hkv, d, 128, (4, 4), bsz * mp, window, max_batch=bsz)
    k, v = _kv(321, bsz, int(lens.max()), hkv, d)
    for b in range(bsz):
        if lens[b] == 0:
            continue
        pair.gpu.append(0, dev_bf16(k[b:b + 1, :lens[b]]), dev_bf16(v[b:b + 1, :lens[b]]),
                        dev_i32(pt[b:b + 1]), dev_i32(np.zeros(1, np.int32)), window_row=b)
        ocache.append(pair.ora, 0, k[b:b + 1, :lens[b]], v[b:b + 1, :lens[b]], pt[b:b + 1],
                      np.zeros(1, np.int32), window_row=b)
    torch.cuda.synchronize()
    assert pair.gpu.get_status() == 0
    assert np.array_equal(pair.gpu.window_host(0), pair.ora.windows[0])
    q = queries(322, 0, bsz, 4 * hkv, d, False)
    pair.decode_check(q, pt, lens)


@pytest.mark.parametrize("window", [0, 16])
def test_decode_steps_cross_pages(window):
    # the step appends its token (quantizing the page it completes once the page
    # is out of the window) and decodes: cache and o as the oracle's append + decode
    bsz, hkv, d, g = 2, 2, 128, 4
    mp = 16
    pt = page_table(330 + window, bsz, mp)
    pair = KpcPair(hkv, d, 128, (4, 2), bsz * mp, window, max_batch=bsz)
    k, v = _kv(331, bsz, 120, hkv, d)
    pair.append(k[:, :70], v[:, :70], pt, np.zeros(bsz, np.int32))
    ws = pair.gpu.workspace(bsz, g * hkv, mp)
    for t in range(70, 120):
        lens = np.full(bsz, t + 1, np.int32)
        q = queries(332 + t, 0, bsz, g * hkv, d, False)
        qd = torch.from_numpy(q).cuda().to(torch.bfloat16)
        o = pair.gpu.decode_step(0, dev_bf16(k[:, t]), dev_bf16(v[:, t]), qd, dev_i32(pt),
                                 dev_i32(lens), workspace=ws)
        written = ocache.append(pair.ora, 0, k[:, t:t + 1], v[:, t:t + 1], pt,
                                np.full(bsz, t, np.int32))
        torch.cuda.synchronize()
        assert pair.gpu.get_status() == 0
        if t % 7 == 0 or any(len(x[0]) for x in written.values()):
            pair.check_written(written, pt)
            ref = attention.decode(pair.gpu_state(), 0, q.astype(np.float64), pt, lens)
            compare_outputs(o.cpu().numpy(), ref)


def test_lossless_grid_equals_exact_attention():
    # keys on per-channel 8-bit grids and values on per-token ones, no rotation:
    # the GPU cache holds K and V exactly, so its attention is plain attention
    # over the inputs (independent of the oracle's quantizer)
    from tests.test_oracle_key_channel import _grid_kv
    bsz, n, hkv, d = 2, 96, 2, 64
    k, v = _grid_kv(41, bsz, n, hkv, d)
    pt = page_table(41, bsz, 8)
    c = kvq.Cache(1, hkv, d, 1, np.full((1, hkv, 2), 8), bsz * 8, 7, bsz, key_per_channel=True)
    c.append(0, dev_bf16(k), dev_bf16(v), dev_i32(pt), dev_i32(np.zeros(bsz, np.int32)))
    q = queries(42, 0, bsz, 4 * hkv, d, True)
    lens = np.full(bsz, n, np.int32)
    o = c.decode(0, torch.from_numpy(q).cuda(), dev_i32(pt), dev_i32(lens))
    torch.cuda.synchronize()
    assert c.get_status() == 0
    compare_outputs(o.cpu().numpy(), attention.exact_decode(q, k, v, lens))


def test_full_size_decode_layer_sampled():
    # the Llama-3-8B-shaped decode layer (batch 16, 32 q / 8 KV heads, d 128,
    # context 4096, K4V4) with per-channel keys, sampled (sequence, head) pairs
    bsz, hkv, hq, d, ctx = 16, 8, 32, 128, 4096
    mp = ctx // 16 + 1
    pt = page_table(350, bsz, mp)
    c = kvq.Cache(1, hkv, d, 128, np.full((1, hkv, 2), 4), bsz * mp, 0, bsz, key_per_channel=True)
    for b in range(0, bsz, 4):
        k, v = _kv(351, 4, ctx, hkv, d, start=0) if b == 0 else _kv(351 + b, 4, ctx, hkv, d)
        c.append(0, dev_bf16(k), dev_bf16(v), dev_i32(pt[b:b + 4]),
                 dev_i32(np.zeros(4, np.int32)), window_row=b)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    q = queries(352, 0, bsz, hq, d, False)
    lens = np.full(bsz, ctx, np.int32)
    o = c.decode(0, torch.from_numpy(q).cuda().to(torch.bfloat16), dev_i32(pt), dev_i32(lens))
    torch.cuda.synchronize()
    st = ocache.CacheState(d, 128, 0, np.full((1, hkv, 2), 4), [c.pool_host(0)],
                           [c.window_host(0)], True)
    pairs = [(0, 0), (3, 7), (8, 2), (15, 5), (11, 1)]
    ref = attention.decode(st, 0, q.astype(np.float64), pt, lens, pairs=pairs)
    compare_outputs(o.cpu().numpy(), ref)

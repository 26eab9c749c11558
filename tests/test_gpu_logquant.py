"""LogQuant mode on the GPU against the oracle (oracle.logquant).

Every token is quantized into the paged cache (codes checked against the
oracle's append); the members of B keep their bf16 K/V in the reserve; decode
attention uses those for B and the codes elsewhere ("LogQuant: Log-Distributed
2-Bit Quantization of KV Cache ...", Methodology sections 2 and 4).  The oracle
runs over the GPU-written pages with the original bf16 values for B, so the
comparison covers the selection, the reserve's bookkeeping across halvings
and the masked decode."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quantized_decode_attention_diag_b300 as kvq
from oracle import cache as ocache, logquant
from tests.parity import compare_outputs, compare_written
from tests.test_gpu_parity import _need_gpu  # noqa: F401
from workloads import kv_tokens, page_table, queries


def _dev(x, dt=torch.bfloat16):
    t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t.to(dt) if dt is not None else t


def _state(c, bits):
    return ocache.CacheState(c.head_dim, c.had_block, 0, np.asarray(bits, np.int64),
                             [c.pool_host(0)], None)


def _check(c, bits, q, pt, lens, k, v, w, q_fp32=False, step=None):
    qd = torch.from_numpy(q).cuda()
    if not q_fp32:
        qd = qd.to(torch.bfloat16)
    if step is None:
        o = c.decode(0, qd, _dev(pt, None), _dev(lens, None))
    else:
        kn, vn = step
        o = c.decode_step(0, _dev(kn), _dev(vn), qd, _dev(pt, None), _dev(lens, None))
    torch.cuda.synchronize()
    assert c.get_status() == 0
    ref = logquant.decode(_state(c, bits), 0, q.astype(np.float64), pt, lens, w, k, v)
    return compare_outputs(o.cpu().numpy(), ref)


def _codes(c, k, v, pt, bsz, lens, hkv, block, bits):
    from oracle import quantizer
    groups = {}
    for b in range(bsz):
        n = int(lens[b])
        for h in range(hkv):
            for kv in (0, 1):
                x = (k if kv == 0 else v)[b, :n, h]
                codes, s, z, u32 = quantizer.rotate_and_quantize(x, block, bits[0][h][kv])
                groups[(b, h, kv)] = (np.arange(n), codes, s, z, u32)
    compare_written(c.pool_host(0), groups, pt, c.head_dim, np.asarray(bits[0]))


@pytest.mark.parametrize("w,bits,d,hkv,g", [(8, (2, 2), 128, 2, 4), (64, (4, 2), 128, 2, 4),
                                            (4, (2, 4), 64, 4, 1), (16, (8, 4), 128, 1, 2)])
def test_prefill_then_decode(w, bits, d, hkv, g):
    lens = np.array([3 * w - 1, 3 * w, 7 * w + 5, 40 * w + 11], np.int32)
    bsz, n = len(lens), int(lens.max())
    mp = (n + 15) // 16
    pt = page_table(70 + w, bsz, mp)
    btab = np.tile(np.array(bits), (1, hkv, 1))
    c = kvq.Cache(1, hkv, d, min(d, 128), btab, bsz * mp, max_batch=bsz, logquant_w=w)
    k = kv_tokens(70 + w, 0, bsz, n, hkv, d, 4, 10.0, 50.0)
    v = kv_tokens(70 + w, 1, bsz, n, hkv, d, 4, 10.0, 50.0)
    for b in range(bsz):       # each sequence its own length, one append each
        c.append(0, _dev(k[b:b + 1, :lens[b]]), _dev(v[b:b + 1, :lens[b]]), _dev(pt[b:b + 1], None),
                 _dev(np.zeros(1, np.int32), None), window_row=b)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    _codes(c, k, v, pt, bsz, lens, hkv, min(d, 128), btab)
    q = queries(70 + w, 0, bsz, g * hkv, d, False)
    _check(c, btab, q, pt, lens, k, v, w)


def test_chunked_prefill_and_steps_across_halvings():
    """Appends in uneven chunks, then decode steps (the new token appended in
    the decode launch) through several halvings; o after every step."""
    w, hkv, d, g, bsz = 8, 2, 128, 4, 3
    bits = np.tile(np.array([4, 2]), (1, hkv, 1))
    n_final = 12 * w + 3
    mp = (n_final + 15) // 16
    pt = page_table(80, bsz, mp)
    c = kvq.Cache(1, hkv, d, 128, bits, bsz * mp, max_batch=bsz, logquant_w=w)
    k = kv_tokens(80, 0, bsz, n_final, hkv, d, 4, 10.0, 50.0)
    v = kv_tokens(80, 1, bsz, n_final, hkv, d, 4, 10.0, 50.0)
    lens = np.zeros(bsz, np.int32)
    for t in (5, 17, 1, 2 * w - 3):       # chunks crossing the first halvings
        c.append(0, _dev(k[:, lens[0]:lens[0] + t]), _dev(v[:, lens[0]:lens[0] + t]),
                 _dev(pt, None), _dev(lens, None))
        lens = lens + t
    torch.cuda.synchronize()
    assert c.get_status() == 0
    q = queries(80, 0, bsz, g * hkv, d, False)
    _check(c, bits, q, pt, lens, k, v, w)
    while lens[0] < n_final:
        lens = lens + 1
        p = int(lens[0]) - 1
        _check(c, bits, q, pt, lens, k, v, w, step=(k[:, p], v[:, p]))
    _codes(c, k, v, pt, bsz, lens, hkv, 128, bits)


def test_reserve_rows_hold_the_members():
    """After a prefill, every member's bf16 K and V sit in its reserve row: the
    ring (row p mod 3W) for the newest members, level buffers for the thinned
    blocks (block b >= 1 in buffer b mod log2 W, block 0 in the last)."""
    w, hkv, d = 16, 2, 64
    a = 4
    n = 9 * w + 7
    mp = (n + 15) // 16
    pt = page_table(90, 1, mp)
    bits = np.full((1, hkv, 2), 2)
    c = kvq.Cache(1, hkv, d, 64, bits, mp, max_batch=1, logquant_w=w)
    k = kv_tokens(90, 0, 1, n, hkv, d, 2, 10.0, 20.0)
    v = kv_tokens(90, 1, 1, n, hkv, d, 2, 10.0, 20.0)
    c.append(0, _dev(k[:, :n - 20]), _dev(v[:, :n - 20]), _dev(pt, None),
             _dev(np.zeros(1, np.int32), None))
    c.append(0, _dev(k[:, n - 20:]), _dev(v[:, n - 20:]), _dev(pt, None),
             _dev(np.array([n - 20], np.int32), None))
    torch.cuda.synchronize()
    res = c.window_host(0)[0]                  # [Hkv][2][rows][d]
    kk = (n - 3 * w) // w + 1
    for p in kvq.kvq_logquant_members(n, w):
        if p >= (kk + 1) * w:
            row = p % (3 * w)
        else:
            blk = p // w
            level = a if blk == 0 else blk % a
            row = 3 * w + level * (w // 2) + (p % w) // 2
        for h in range(hkv):
            assert np.array_equal(res[h, 0, row], k[0, p, h]), (p, h)
            assert np.array_equal(res[h, 1, row], v[0, p, h]), (p, h)


def test_decode_split_limit_with_reserve():
    # one sequence, one KV head (4 query heads), 65536 tokens, W = 128, K2V2: the
    # wave leaves the unit all 592 slots, so it takes 256 splits of 16 pages and
    # four reserve CTAs -- 260 partials, the ticket combine's largest count
    w, d, hkv, g, n = 128, 128, 1, 4, 65536
    mp = n // 16
    pt = page_table(93, 1, mp)
    btab = np.array([[[2, 2]]])
    c = kvq.Cache(1, hkv, d, 128, btab, mp, max_batch=1, logquant_w=w)
    k = kv_tokens(93, 0, 1, n, hkv, d, 4, 10.0, 50.0)
    v = kv_tokens(93, 1, 1, n, hkv, d, 4, 10.0, 50.0)
    c.append(0, _dev(k), _dev(v), _dev(pt, None), _dev(np.zeros(1, np.int32), None),
             window_row=0)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    q = queries(93, 0, 1, g * hkv, d, False)
    _check(c, btab, q, pt, np.array([n], np.int32), k, v, w)

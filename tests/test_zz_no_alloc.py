"""kvq_decode_attn_static: decode without a caller-provided workspace.

This entry point serves callers that may not allocate device memory (a plugin
whose host process owns every device byte, or a path that must never reach
cudaMalloc because it can synchronise the device).  It must give the same
result as kvq_decode_attn with a workspace, on consecutive calls that reuse
the library's fixed scratch, and refuse sizes beyond that scratch.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test.  It builds its own inputs and needs
no earlier test: it passes alone in a fresh process too.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quantized_decode_attention_diag_b300 as kvq
from tests.parity import O_MAX_ABS, O_MEAN_ABS
from workloads import kv_tokens, page_table, queries


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_attention_diag_b300 import build
    build.build()


def _cache(bsz, ctx, window=0, seed=90, fill=True):
    hkv, d = 8, 128
    mp = (ctx + 15) // 16
    pt = page_table(seed, bsz, mp)
    c = kvq.Cache(1, hkv, d, 128, np.tile(np.array([4, 2]), (1, hkv, 1)), bsz * mp,
                  window=window, max_batch=max(bsz, 1))
    if not fill:
        return c, torch.from_numpy(pt).cuda()
    k = kv_tokens(seed, 0, bsz, ctx, hkv, d, 4, 10.0, 50.0)
    v = kv_tokens(seed, 1, bsz, ctx, hkv, d, 4, 10.0, 50.0)
    dev = lambda x: torch.from_numpy(x).cuda()
    c.append(0, dev(k).to(torch.bfloat16), dev(v).to(torch.bfloat16), dev(pt),
             dev(np.zeros(bsz, np.int32)))
    return c, dev(pt)


def _both(c, pt, q, lens):
    bsz, hq, d = q.shape
    ref = c.decode(0, q, pt, lens)
    out = torch.full((bsz, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_attn_static(c.desc, 0, q, False, pt, int(pt.shape[1]), lens, bsz, hq, 0.0, out)
    torch.cuda.synchronize()
    assert c.get_status() == 0
    diff = (out - ref).abs()
    assert torch.isfinite(out).all()
    assert diff.max().item() <= O_MAX_ABS and diff.mean().item() <= O_MEAN_ABS
    return out


def test_static_workspace_matches_workspace_entry_on_consecutive_calls():
    c, pt = _cache(4, 700, window=64)
    q1 = torch.from_numpy(queries(91, 0, 4, 32, 128, False)).cuda().to(torch.bfloat16)
    q2 = torch.from_numpy(queries(91, 1, 4, 32, 128, False)).cuda().to(torch.bfloat16)
    l1 = torch.tensor([700, 1, 333, 64], dtype=torch.int32, device="cuda")
    l2 = torch.tensor([650, 700, 129, 0], dtype=torch.int32, device="cuda")
    o1 = _both(c, pt, q1, l1)           # first call: the scratch is fresh
    o2 = _both(c, pt, q2, l2)           # second call: it holds the first call's contents
    assert not torch.equal(o1, o2)


def test_static_workspace_rejects_oversized_decodes():
    bsz = 600                            # 4800 (sequence, KV head) pairs: above 8 MiB of scratch
    c, pt = _cache(bsz, 16, seed=92, fill=False)   # rejected before any launch
    need = kvq.kvq_decode_workspace_bytes(c.desc, bsz, 32, int(pt.shape[1]))
    assert need > kvq.STATIC_WORKSPACE_BYTES
    q = torch.zeros((bsz, 32, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((bsz, 32, 128), dtype=torch.float32, device="cuda")
    lens = torch.full((bsz,), 16, dtype=torch.int32, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attn_static(c.desc, 0, q, False, pt, int(pt.shape[1]), lens, bsz, 32, 0.0, o)
    assert e.value.status == kvq.KVQ_EWORKSPACE
    assert "fixed" in kvq.kvq_last_error()
    torch.cuda.synchronize()
    assert (o == 0).all()                # nothing was launched


def test_static_with_overlap_flag():
    """With KVQ_LAUNCH_OVERLAP set in the descriptor, the static entry point
    gives the result of an ordinary launch, bit for bit, on calls that follow
    each other on one stream.  (Each call clears its tickets with a memset
    first, and a memset orders the decode after the previous kernel as usual,
    so these decodes never actually overlap: the test checks that the flag
    changes nothing, not the overlap itself, which the ordinary entry point's
    tests cover.)"""
    c, pt = _cache(4, 2000, seed=94)
    bsz, hq, d = 4, 32, 128
    q = torch.from_numpy(queries(94, 0, bsz, hq, d, False)).cuda().to(torch.bfloat16)
    lens = torch.from_numpy(np.array([2000, 1, 777, 1600], np.int32)).cuda()
    outs = []
    for flags in (0, kvq.LAUNCH_OVERLAP):
        c.desc.launch_flags = flags
        o = [torch.full((bsz, hq, d), float("nan"), dtype=torch.float32, device="cuda")
             for _ in range(3)]
        for x in o:      # back to back on one stream
            kvq.kvq_decode_attn_static(c.desc, 0, q, False, pt, int(pt.shape[1]), lens, bsz,
                                       hq, 0.0, x)
        torch.cuda.synchronize()
        assert c.get_status() == 0
        assert torch.equal(o[0], o[1]) and torch.equal(o[1], o[2])
        outs.append(o[0])
    c.desc.launch_flags = 0
    assert torch.equal(outs[0], outs[1])

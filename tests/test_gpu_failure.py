"""Failure detection on the GPU without a fault.

The decode's main loop gives up on a page copy after a bounded wait (about a
second), records KVQ_DEV_COPY_TIMEOUT in the cache's status word, waits --
with the full limit -- for every copy it issued, and returns; the context
stays usable.  Here a child process shortens the wait to ~1 cycle through
the debug variable KVQ_DEBUG_COPY_WAIT_LOG2 (read once per process), so that
waits on copies of valid memory, which do complete, run out: the call must
return, the status bit must be set, and the same process must go on to run
an ordinary decode after clearing the status."""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import quantized_decode_attention_diag_b300 as kvq
from workloads import kv_tokens, page_table, queries
bsz, hkv, d, ctx = 4, 8, 128, 2048
mp = ctx // 16
c = kvq.Cache(1, hkv, d, 128, np.full((1, hkv, 2), 4), bsz * mp)
k = torch.from_numpy(kv_tokens(7, 0, bsz, ctx, hkv, d, 4, 10.0, 50.0)).cuda().to(torch.bfloat16)
v = torch.from_numpy(kv_tokens(7, 1, bsz, ctx, hkv, d, 0, 10.0, 50.0)).cuda().to(torch.bfloat16)
pt = torch.from_numpy(page_table(7, bsz, mp)).cuda()
c.append(0, k, v, pt, torch.zeros(bsz, dtype=torch.int32, device="cuda"))
torch.cuda.synchronize()
assert c.get_status() == 0
q = torch.from_numpy(queries(7, 0, bsz, 32, d, False)).cuda().to(torch.bfloat16)
lens = torch.full((bsz,), ctx, dtype=torch.int32, device="cuda")
timeouts = 0
for _ in range(20):
    c.reset_status()
    o = c.decode(0, q, pt, lens)
    torch.cuda.synchronize()
    st = c.get_status()
    assert st & ~kvq.DEV_COPY_TIMEOUT == 0, hex(st)
    timeouts += bool(st & kvq.DEV_COPY_TIMEOUT)
# the context is still usable: plain device work, and a status that clears
c.reset_status()
torch.cuda.synchronize()
assert c.get_status() == 0
assert float((torch.ones(1000, device="cuda") * 2).sum()) == 2000.0
print("TIMEOUTS", timeouts)
'''


def _run(env_value):
    env = dict(os.environ)
    if env_value is None:
        env.pop("KVQ_DEBUG_COPY_WAIT_LOG2", None)
    else:
        env["KVQ_DEBUG_COPY_WAIT_LOG2"] = env_value
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    return int(r.stdout.split("TIMEOUTS")[-1])


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_decode_attention_diag_b300 import build
    build.build()


def test_short_copy_wait_reports_timeout_and_returns():
    assert _run("0") > 0


def test_default_copy_wait_never_times_out():
    assert _run(None) == 0

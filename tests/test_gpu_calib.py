"""Distortion calibration (kvq_distortion) against the oracle's measure_mse,
and the calibrate -> fit -> allocate pipeline.

The GPU takes every code decision by the oracle's rule (fp32 difference and
reciprocal, round-half-even of the exact product), so the two MSEs differ only
by the fp32 rounding of c s + z and of the sums: relative 1e-5."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quantized_decode_attention_diag_b300 as kvq
from oracle import allocator, distortion
from tests.test_gpu_parity import _need_gpu  # noqa: F401
from workloads import kv_tokens

RTOL = 1e-5


def _gpu_mse(x, d, block, widths):
    X = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(torch.bfloat16)
    out = kvq.kvq_distortion(d, block, X, widths)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("d,block", [(128, 128), (128, 64), (128, 32), (64, 64), (64, 32)])
@pytest.mark.parametrize("t", [1, 37, 1000])
def test_mse_matches_oracle(d, block, t):
    hkv, widths = 3, [1, 2, 3, 4, 5, 6, 7, 8]
    x = kv_tokens(300 + t, 0, 1, t, hkv, d, 4, 10.0, 50.0)[0]        # [t][hkv][d], bf16-exact
    got = _gpu_mse(x, d, block, widths)
    for h in range(hkv):
        want = distortion.measure_mse(x[:, h], block, widths)
        np.testing.assert_allclose(got[h], want, rtol=RTOL, atol=0)


def test_mse_empty_and_constant_inputs():
    X = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = kvq.kvq_distortion(128, 128, X, [2, 4])
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0
    # constant vectors whose value is fp16-exact after rotation: s = 0, no error
    x = np.zeros((50, 2, 128), np.float32)
    x[:, :, 0] = 1.0                                  # rotation: every u_j = 1
    got = _gpu_mse(x, 128, 128, [2, 4, 8])
    assert np.all(got == 0.0)


def test_calibrate_fit_allocate_pipeline():
    """Per-(layer, head, K|V) MSE on calibration sequences -> (alpha, beta) ->
    the greedy allocation, against the oracle's MSE and fit on the same data."""
    L, hkv, d, t, widths = 4, 4, 128, 512, [2, 3, 4, 5, 6]
    mse_gpu, mse_ora = [], []
    for l in range(L):
        for kv in range(2):
            # K with outlier channels, V plain: different distortion curves
            x = kv_tokens(400 + l, kv, 1, t, hkv, d, 4 if kv == 0 else 0, 10.0, 50.0)[0]
            mse_gpu.append(_gpu_mse(x, d, 128, widths))
            mse_ora.append(np.stack([distortion.measure_mse(x[:, h], 128, widths)
                                     for h in range(hkv)]))
    # component order (layer * Hkv + head) * 2 + kv
    g = np.stack(mse_gpu).reshape(L, 2, hkv, -1).transpose(0, 2, 1, 3).reshape(-1, len(widths))
    o = np.stack(mse_ora).reshape(L, 2, hkv, -1).transpose(0, 2, 1, 3).reshape(-1, len(widths))
    np.testing.assert_allclose(g, o, rtol=RTOL)
    alpha, beta = kvq.kvq_fit_distortion(g, widths)
    for i in range(g.shape[0]):
        a, b = distortion.fit(widths, o[i])
        assert abs(alpha[i] / a - 1) < 1e-3 and abs(beta[i] / b - 1) < 1e-4
        assert 3.0 < beta[i] < 6.0          # RateQuant prints 3.6 .. 5.3 for real quantizers
    sens = np.random.default_rng(5).lognormal(0.0, 1.0, size=g.shape[0])
    n = g.shape[0]
    budget = int(3.5 * n)
    allowed = [[4, 8] if i % 2 == 0 else [2, 4] for i in range(n)]
    bits, left = kvq.kvq_alloc_bits(sens * alpha, beta, budget, [kvq.mask_of(a) for a in allowed])
    want, wleft = allocator.greedy(sens * alpha, beta, budget, allowed)
    assert bits == list(want) and left == wleft

"""Pins for oracle.hadamard (block-diagonal Walsh-Hadamard rotation)."""
import numpy as np
import pytest

from oracle import hadamard
from tests.conftest import GOLDEN


def _golden_h8():
    rows = [l.split() for l in open(f"{GOLDEN}/hadamard_sylvester_8.txt")
            if l.strip() and not l.startswith("#")]
    return np.array(rows, dtype=np.int64)


def test_h8_matches_hand_written_matrix():
    assert np.array_equal(hadamard.sylvester(8), _golden_h8())


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128])
def test_orthogonality_and_symmetry(n):
    h = hadamard.sylvester(n)
    assert np.array_equal(h @ h.T, n * np.eye(n, dtype=np.int64))
    assert np.array_equal(h, h.T)


@pytest.mark.parametrize("n", [32, 64, 128])
def test_entries_are_popcount_signs(n):
    h = hadamard.sylvester(n)
    for i in range(n):
        for j in range(n):
            assert h[i, j] == (-1) ** bin(i & j).count("1")


def _fwht_recursive(x):
    """Hadamard product by the Sylvester recursion on vectors (independent path)."""
    n = len(x)
    if n == 1:
        return list(x)
    a = _fwht_recursive(x[: n // 2])
    b = _fwht_recursive(x[n // 2:])
    return [p + q for p, q in zip(a, b)] + [p - q for p, q in zip(a, b)]


@pytest.mark.parametrize("d,n", [(64, 64), (64, 32), (128, 128), (128, 64), (128, 32)])
def test_rotate_is_block_diagonal_fwht(d, n):
    rng = np.random.default_rng(d + n)
    x = rng.standard_normal((3, d))
    u = hadamard.rotate(x, n)
    for r in range(3):
        want = []
        for blk in range(d // n):
            want += _fwht_recursive(list(x[r, blk * n:(blk + 1) * n]))
        assert np.allclose(u[r], want, rtol=0, atol=1e-12)
    hb = hadamard.block_hadamard(d, n)
    off = np.ones((d, d), bool)
    for blk in range(d // n):
        off[blk * n:(blk + 1) * n, blk * n:(blk + 1) * n] = False
    assert not hb[off].any()


@pytest.mark.parametrize("n", [32, 64, 128])
def test_inner_product_preserved(n):
    # q . k = (H q) . (H k) / n  (the once-rotated query scores rotated keys)
    rng = np.random.default_rng(n)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    hq, hk = hadamard.rotate(q, n), hadamard.rotate(k, n)
    assert abs(hq @ hk / n - q @ k) < 1e-12 * max(1.0, abs(q @ k)) * 10
    r = hadamard.orthonormal(128, n)
    assert abs(np.linalg.norm(r @ q) - np.linalg.norm(q)) < 1e-12
    assert np.allclose(hadamard.unrotate(hadamard.rotate(q, n), n), q, atol=1e-13)


def test_rejects_bad_sizes():
    with pytest.raises(ValueError):
        hadamard.sylvester(12)
    with pytest.raises(ValueError):
        hadamard.block_hadamard(96, 64)

"""Pins for oracle.layout: hand-packed bytes, page sizes, write/read round trip."""
import numpy as np
import pytest

from oracle import layout
from tests.conftest import golden_rows


@pytest.mark.parametrize("row", golden_rows("layout_pack_examples.txt"))
def test_pack_examples(row):
    bits = int(row[0])
    codes = np.array(row[1].split(), dtype=np.uint8)
    want = bytes.fromhex("".join(row[2].split()))
    assert layout.pack(codes, bits).tobytes() == want
    assert np.array_equal(layout.unpack(np.frombuffer(want, np.uint8), bits, len(codes)), codes)


def test_page_bytes():
    assert layout.page_bytes(128, np.array([[4, 4]] * 8)) == 17408
    assert layout.page_bytes(128, np.array([[4, 2]] * 8)) == 13312
    assert layout.page_bytes(64, np.array([[4, 2]] * 4)) == 3584
    offs = layout.head_offsets(128, np.array([[4, 2], [8, 4], [4, 4]]))
    assert offs.tolist() == [0, 16 * (64 + 32 + 8), 16 * (64 + 32 + 8) + 16 * (128 + 64 + 8)]
    assert all(o % 16 == 0 for o in offs)


def test_write_read_round_trip():
    bits = np.array([[4, 2], [8, 4]])
    pool = np.zeros((3, layout.page_bytes(64, bits)), np.uint8)
    view = layout.PageView(pool, 64, bits)
    rng = np.random.default_rng(0)
    for h in range(2):
        for kv in range(2):
            b = bits[h, kv]
            codes = rng.integers(0, 1 << b, size=(5, 64)).astype(np.uint8)
            s = rng.random(5).astype(np.float16)
            z = (-rng.random(5)).astype(np.float16)
            pages, slots = np.array([0, 2, 1, 2, 0]), np.array([0, 15, 7, 3, 9])
            view.write_many(pages, slots, h, kv, codes, s, z)
            c2, s2, z2 = view.read(pages, slots, h, kv)
            assert np.array_equal(c2, codes) and np.array_equal(s2, s) and np.array_equal(z2, z)

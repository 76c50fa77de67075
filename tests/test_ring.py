"""Local-window page recycling, host side: the ring length and the block-table rows.

For random windows, page sizes, call sizes and lengths, every page a call touches
(decode: [L - W, L); prefill of n tokens on prefix L - n: [max(0, L - n + 1 - W), L);
append of n tokens: [L - n, L)) must be mapped, freed and unwritten pages must be -1,
and no two mapped pages of one sequence may share a ring slot.  These are properties
of the positions alone, checked here by brute force over the positions.
"""
import numpy as np
import pytest

cai = pytest.importorskip("int8_mqa_decode_gb300")


def _lib_or_skip():
    try:
        cai.load()
    except Exception as e:  # library not built on this machine
        pytest.skip(f"libcai not loadable: {e}")


def test_ring_pages_formula():
    _lib_or_skip()
    assert cai.cai_ring_pages(1024, 16, 1) == 65
    assert cai.cai_ring_pages(1024, 16, 256) == 81
    assert cai.cai_ring_pages(1024, 64, 1) == 17
    assert cai.cai_ring_pages(1, 16, 1) == 2
    assert cai.cai_ring_pages(16, 16, 1) == 2
    assert cai.cai_ring_pages(17, 16, 1) == 3
    for bad in [(0, 16, 1), (1024, 0, 1), (1024, 16, 0), (-5, 16, 1)]:
        assert cai.cai_ring_pages(*bad) == 0


def test_ring_table_row_contents():
    _lib_or_skip()
    ids = np.arange(100, 105, dtype=np.int32)  # ring of 5
    row = cai.cai_ring_table_row(ids, hi=70, page_size=16, max_pages_per_seq=8)  # pages 0..4 written
    assert row.tolist() == [100, 101, 102, 103, 104, -1, -1, -1]
    row = cai.cai_ring_table_row(ids, hi=113, page_size=16, max_pages_per_seq=10)  # pages 0..7, last 5 live
    assert row.tolist() == [-1, -1, -1, 103, 104, 100, 101, 102, -1, -1]
    row = cai.cai_ring_table_row(ids, hi=0, page_size=16, max_pages_per_seq=4)
    assert row.tolist() == [-1, -1, -1, -1]
    with pytest.raises(cai.CaiError):
        cai.cai_ring_table_row(ids, hi=200, page_size=16, max_pages_per_seq=8)  # beyond the table
    with pytest.raises(cai.CaiError):
        cai.cai_ring_table_row(ids, hi=-1, page_size=16, max_pages_per_seq=8)


def _touched(lo, hi, P):
    return set(range(lo // P, (hi - 1) // P + 1)) if hi > lo else set()


@pytest.mark.parametrize("seed", range(4))
def test_ring_covers_every_call(seed):
    _lib_or_skip()
    rng = np.random.default_rng(seed)
    for _ in range(200):
        P = int(rng.choice([16, 32, 64]))
        W = int(rng.integers(1, 3000))
        n = int(rng.choice([1, 1, 7, 64, 256]))
        L = int(rng.integers(n, 20000))
        R = cai.cai_ring_pages(W, P, n)
        mp = (L + P - 1) // P + int(rng.integers(0, 4))
        ids = rng.permutation(10 * R)[:R].astype(np.int32)
        row = cai.cai_ring_table_row(ids, L, P, mp)
        live = {k for k in range(mp) if row[k] >= 0}
        # every page of every call ending at L is mapped
        for lo in (max(0, L - W), max(0, L - n + 1 - W), L - n):
            assert _touched(lo, L, P) <= live, (P, W, n, L)
        # nothing beyond the written positions, and no more than the ring
        assert max(live) == (L - 1) // P and len(live) == min(R, (L + P - 1) // P)
        # one slot per live page, the slot of logical page k
        assert len({int(row[k]) for k in live}) == len(live)
        assert all(row[k] == ids[k % R] for k in live)

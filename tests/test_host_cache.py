"""Cross-turn host KV cache (radix tree over whole pages, rolling hash with
token confirmation, LRU leaf eviction): host-memory pools, no GPU needed."""
import numpy as np
import pytest

import int8_mqa_decode_gb300 as cai
from int8_mqa_decode_gb300 import build as cai_build

P = 16
PB = 16 * 264


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cai_build.build()
    cai.load()


class HostPool:
    """A pool in host memory (numpy), described by the C struct."""

    def __init__(self, num_pages, seed=None):
        rng = np.random.default_rng(seed)
        self.buf = rng.integers(0, 256, size=num_pages * PB, dtype=np.uint8) if seed is not None else \
            np.zeros(num_pages * PB, dtype=np.uint8)
        self.struct = cai.cai_kv_pool(self.buf.ctypes.data, num_pages, P, 128)

    def page(self, i):
        return self.buf[i * PB:(i + 1) * PB]


def tokens(seed, n):
    return np.random.default_rng(seed).integers(0, 50000, size=n).astype(np.int32)


def test_store_match_restore_bit_identical():
    c = cai.cai_host_cache_create(P, 2, 32)
    try:
        src = [HostPool(20, seed=1), HostPool(20, seed=2)]
        a = tokens(3, 5 * P + 7)                      # 5 full pages + a partial one (ignored)
        table = np.array([3, 7, 1, 12, 9, 4], dtype=np.int32)
        cai.cai_host_cache_store(c, a, [p.struct for p in src], table)
        assert cai.cai_host_cache_match(c, a) == 5 * P
        b = a.copy()
        b[3 * P + 2] += 1                             # diverges inside page 3: three pages shared
        assert cai.cai_host_cache_match(c, b) == 3 * P
        assert cai.cai_host_cache_match(c, tokens(4, 3 * P)) == 0
        dst = [HostPool(8), HostPool(8)]
        new_table = np.array([5, 0, 6], dtype=np.int32)
        cai.cai_host_cache_restore(c, b, 3 * P, [p.struct for p in dst], new_table)
        for buf in range(2):
            for k in range(3):
                assert np.array_equal(dst[buf].page(new_table[k]), src[buf].page(table[k]))
            assert not dst[buf].page(1).any()         # untouched
        s = cai.cai_host_cache_stats(c)
        assert s["hits"] == 2 and s["misses"] == 1 and s["pages_cached"] == 5 and s["evictions"] == 0
    finally:
        cai.cai_host_cache_destroy(c)


def test_lru_evicts_leaves_and_keeps_paths_whole():
    c = cai.cai_host_cache_create(P, 1, 6)
    try:
        src = [HostPool(30, seed=5)]
        a, b = tokens(10, 4 * P), tokens(11, 4 * P)
        cai.cai_host_cache_store(c, a, [src[0].struct], np.arange(4, dtype=np.int32))
        cai.cai_host_cache_store(c, b, [src[0].struct], np.arange(10, 14, dtype=np.int32))
        # 8 pages wanted, 6 slots: a (least recent) lost its last two pages, leaf first.
        assert cai.cai_host_cache_match(c, b) == 4 * P
        assert cai.cai_host_cache_match(c, a) == 2 * P
        assert cai.cai_host_cache_stats(c)["evictions"] == 2
        # A shared prefix is stored once: a continuation of b reuses b's pages.
        b2 = np.concatenate([b, tokens(12, P)])
        cai.cai_host_cache_store(c, b2, [src[0].struct], np.arange(10, 15, dtype=np.int32))
        assert cai.cai_host_cache_match(c, b2) == 5 * P
        assert cai.cai_host_cache_stats(c)["pages_cached"] == 6
        # Restoring what is no longer cached is refused, and nothing is written.
        dst = HostPool(8)
        with pytest.raises(cai.CaiError):
            cai.cai_host_cache_restore(c, a, 4 * P, [dst.struct], np.arange(4, dtype=np.int32))
        assert not dst.buf.any()
    finally:
        cai.cai_host_cache_destroy(c)


def test_path_longer_than_capacity_is_refused():
    c = cai.cai_host_cache_create(P, 1, 3)
    try:
        pool = HostPool(8, seed=1)
        with pytest.raises(cai.CaiError) as e:
            cai.cai_host_cache_store(c, tokens(20, 5 * P), [pool.struct], np.arange(5, dtype=np.int32))
        assert e.value.status == 3
    finally:
        cai.cai_host_cache_destroy(c)


def test_restore_batch_equals_restores():
    """Several sequences restored in one call land byte for byte where per-sequence restores
    put them; a sequence that is not fully cached rejects the whole batch (nothing copied)."""
    c = cai.cai_host_cache_create(P, 1, 64)
    try:
        src = [HostPool(40, seed=11)]
        seqs = [tokens(20 + i, (3 + i) * P) for i in range(3)]
        rows = [np.arange(10 * i, 10 * i + 8, dtype=np.int32) for i in range(3)]
        for s, r in zip(seqs, rows):
            cai.cai_host_cache_store(c, s, [p.struct for p in src], r)
        one = [HostPool(40)]
        two = [HostPool(40)]
        dst_rows = [np.arange(30 - 10 * i, 38 - 10 * i, dtype=np.int32) for i in range(3)]
        for s, r in zip(seqs, dst_rows):
            cai.cai_host_cache_restore(c, s, len(s), [p.struct for p in one], r)
        cai.cai_host_cache_restore_batch(c, seqs, [len(s) for s in seqs], [p.struct for p in two], dst_rows)
        assert np.array_equal(one[0].buf, two[0].buf) and one[0].buf.any()
        three = [HostPool(40)]
        missing = tokens(99, 2 * P)
        with pytest.raises(cai.CaiError):
            cai.cai_host_cache_restore_batch(c, seqs + [missing], [len(s) for s in seqs] + [2 * P],
                                             [p.struct for p in three], dst_rows + [dst_rows[0]])
        assert not three[0].buf.any()
    finally:
        cai.cai_host_cache_destroy(c)

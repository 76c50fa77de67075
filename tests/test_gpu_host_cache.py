"""Cross-turn host KV cache on the GPU: pages stored from device pools and
restored into other pages of a fresh pool are byte-identical, and decoding a
resumed dialogue over the restored prefix gives the same bits as decoding the
original cache."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import harness  # noqa: E402
import int8_mqa_decode_gb300 as cai  # noqa: E402
import synth  # noqa: E402


def test_restore_device_pages_and_resume_decode():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_mqa_decode_gb300 import build
    build.build()
    P = 16
    L = 300
    w = synth.Workload("dialogue", 1, 8, P, np.array([L]), [0], [0], seed=77)
    orig = harness.PagedCache(w)
    orig.fill(upto=w.ctx_len)
    torch.cuda.synchronize()
    tokens = np.arange(1000, 1000 + L, dtype=np.int32)  # the dialogue's token ids
    cache = cai.cai_host_cache_create(P, 1, 64)
    try:
        cai.cai_host_cache_store(cache, tokens, orig.pools, orig.table_np[0])
        n = cai.cai_host_cache_match(cache, tokens)
        assert n == (L // P) * P
        # A fresh pool with a different page placement: restore the prefix, append the rest.
        fresh = harness.PagedCache(w, sentinel=0)
        fresh.table_np[0, : (L + P - 1) // P] = fresh.table_np[0, : (L + P - 1) // P][::-1]
        fresh.table = torch.from_numpy(fresh.table_np).cuda()
        cai.cai_host_cache_restore(cache, tokens, n, fresh.pools, fresh.table_np[0])
        torch.cuda.synchronize()
        for k in range(n // P):
            a = orig.pools[0].pages.view(-1, cai.cai_page_bytes(P))[orig.table_np[0, k]]
            b = fresh.pools[0].pages.view(-1, cai.cai_page_bytes(P))[fresh.table_np[0, k]]
            assert torch.equal(a, b)
        import synth.gpu as sgpu
        k_t = torch.empty(1, L - n, 128, device="cuda")
        v_t = torch.empty_like(k_t)
        sgpu.normal_rows(k_t, w.seed, synth.stream_k(0), 0, p_const=n)
        sgpu.normal_rows(v_t, w.seed, synth.stream_v(0), 0, p_const=n)
        cai.cai_kv_append(fresh.pools[0], k_t, v_t, fresh.table, torch.tensor([n], dtype=torch.int32, device="cuda"))
        q = orig.decode_q(0)
        o1 = torch.empty(1, 8, 128, device="cuda")
        o2 = torch.empty_like(o1)
        orig.decode(0, q, o1)
        fresh.decode(0, q, o2)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    finally:
        cai.cai_host_cache_destroy(cache)

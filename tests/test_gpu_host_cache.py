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


def test_dialogue_turn_restore_then_prefill_matches_oracle():
    """The cross-turn flow end to end: turn 1 of a dialogue (300 tokens) is cached in host
    memory; turn 2 (400 tokens) restores the longest cached prefix (whole pages, 288 tokens)
    into a fresh pool with another page placement, appends the remaining 112 tokens and runs
    cai_mqa_prefill_chunk over them; every new token's output and lse against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_mqa_decode_gb300 import build
    build.build()
    import oracle
    import synth.gpu  # noqa: F401
    synth.gpu.build()
    P, Hq, L1, L2, seed = 16, 8, 300, 400, 91
    tokens = np.arange(5000, 5000 + L2, dtype=np.int32)  # the dialogue's token ids
    turn1 = synth.Workload("turn1", 1, Hq, P, np.array([L1]), [0, 0], [0, 1], seed=seed)
    first = harness.PagedCache(turn1)
    first.fill(upto=turn1.ctx_len)
    torch.cuda.synchronize()
    cache = cai.cai_host_cache_create(P, 2, 64)
    try:
        cai.cai_host_cache_store(cache, tokens[:L1], first.pools, first.table_np[0])
        n = cai.cai_host_cache_match(cache, tokens)
        assert n == (L1 // P) * P == 288
        turn2 = synth.Workload("turn2", 1, Hq, P, np.array([L2]), [0, 0], [0, 1], n_new=L2 - n, seed=seed)
        fresh = harness.PagedCache(turn2, sentinel=0x5A)
        pages = (L2 + P - 1) // P
        fresh.table_np[0, :pages] = fresh.table_np[0, :pages][::-1]  # another placement
        fresh.table = torch.from_numpy(fresh.table_np).cuda()
        cai.cai_host_cache_restore(cache, tokens, n, fresh.pools, fresh.table_np[0])
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        fresh.append_step(err=err)  # positions n .. L2-1 of both buffers
        q = fresh.prefill_q()
        out = torch.full((1, L2 - n, Hq, 128), float("nan"), device="cuda")
        lse = torch.full((1, L2 - n, Hq), float("nan"), device="cuda")
        fresh.prefill(q, out, lse, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for k in range(n // P):  # restored pages are byte-identical, in both buffers
            for buf in range(2):
                a = first.pools[buf].pages.view(-1, cai.cai_page_bytes(P))[first.table_np[0, k]]
                b = fresh.pools[buf].pages.view(-1, cai.cai_page_bytes(P))[fresh.table_np[0, k]]
                assert torch.equal(a, b)
        kc, ks, vc, vs = oracle.seq_kv(seed, 0, 0, L2)
        qb = synth.q_rows(seed, synth.STREAM_Q_PREFILL, 0, (L2 - n) * Hq).reshape(L2 - n, Hq, 128)
        ref, ref_lse = oracle.prefill_seq(qb, kc, ks, vc, vs, n, 0, turn2.softmax_scale)
        assert np.abs(out.cpu().numpy()[0] - ref).max() <= 2e-3
        assert np.abs(lse.cpu().numpy()[0] - ref_lse).max() <= 2e-3
    finally:
        cai.cai_host_cache_destroy(cache)

"""GPU parity of grouped-query decode: num_kv_heads pools, each read by its group of
query heads, against the oracle's MQA attention of every group over its own KV head;
num_kv_heads = 1 equals the MQA entry point bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import harness  # noqa: E402
import int8_mqa_decode_gb300 as cai  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_mqa_decode_gb300 import build
    build.build()
    import synth.gpu
    synth.gpu.build()


def gqa_case(Hkv, Hq, L, P=16, window=0, num_splits=0, seed=81):
    # One "buffer" per KV head: the harness fills each pool from its own seeded stream.
    L = np.asarray(L, dtype=np.int64)
    w = synth.Workload("gqa", len(L), Hq, P, L, [window] * Hkv, list(range(Hkv)), n_new=1, seed=seed)
    cache = harness.PagedCache(w)
    cache.fill()
    cache.append_step()
    q = cache.decode_q(0)
    out = torch.full((w.batch, Hq, 128), float("nan"), device="cuda")
    lse = torch.full((w.batch, Hq), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(cai.cai_gqa_decode_workspace_size(w.batch, Hq, Hkv, cache.max_pages_per_seq, P, window,
                                                       num_splits), dtype=torch.uint8, device="cuda")
    cai.cai_gqa_decode(cache.pools, q, cache.table, cache.ctx_len, window, w.softmax_scale, num_splits, ws, out, lse,
                       err)
    torch.cuda.synchronize()
    return w, cache, q, out.cpu().numpy(), lse.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("Hkv,Hq,window,splits", [(8, 64, 0, 0), (4, 32, 0, 3), (2, 128, 0, 0), (8, 8, 512, 0),
                                                  (4, 64, 1024, 2)])
def test_gqa_decode_matches_oracle(Hkv, Hq, window, splits):
    L = [1, 700, 4096, 2049, 130]
    w, cache, q, out, lse, err = gqa_case(Hkv, Hq, L, window=window, num_splits=splits)
    assert err == 0
    G = Hq // Hkv
    for b in range(w.batch):
        qb = synth.q_rows(w.seed, synth.stream_q(0), b, Hq)
        for j in range(Hkv):
            kc, ks, vc, vs = oracle.seq_kv(w.seed, j, b, int(w.ctx_len[b]))
            o_ref, l_ref = oracle.decode_seq(qb[j * G:(j + 1) * G], kc, ks, vc, vs, int(w.ctx_len[b]), window,
                                             w.softmax_scale)
            assert np.abs(out[b, j * G:(j + 1) * G] - o_ref).max() <= ATOL, (b, j)
            assert np.abs(lse[b, j * G:(j + 1) * G] - l_ref).max() <= ATOL, (b, j)


def test_gqa_one_kv_head_is_mqa():
    w, cache, q, out, lse, err = gqa_case(1, 32, [300, 5000, 17], seed=83)
    assert err == 0
    o2 = torch.empty(w.batch, 32, 128, device="cuda")
    l2 = torch.empty(w.batch, 32, device="cuda")
    cache.decode(0, q, o2, l2)
    torch.cuda.synchronize()
    assert np.array_equal(out, o2.cpu().numpy()) and np.array_equal(lse, l2.cpu().numpy())


def test_gqa_footprint_ratio():
    # Bytes of KV per token: one head for MQA against num_kv_heads for GQA (the pages' 8X at 8 KV heads).
    mqa = cai.cai_page_bytes(16) // 16
    assert mqa == 264
    assert 8 * mqa == 2112

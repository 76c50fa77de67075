"""GPU parity of local-window page recycling: local buffers hold each sequence in a
ring of cai_ring_pages() pages, table entries of freed and unwritten pages are -1,
and decode and windowed prefill must match the oracle (which keeps every position)
without ever reading a freed page (any such read sets CAI_DEVERR_PAGE)."""
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


def decode_errs(cache, layer):
    w = cache.w
    q = cache.decode_q(layer)
    out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), device="cuda")
    lse = torch.full((w.batch, w.num_q_heads), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.decode(layer, q, out, lse, err=err)
    torch.cuda.synchronize()
    return int(err.item()), out.cpu().numpy(), lse.cpu().numpy()


def check_decode(cache, layer, out, lse):
    w = cache.w
    for b in range(w.batch):
        L = int(w.ctx_len[b])
        buf = w.layer_to_buffer[layer]
        kc, ks, vc, vs = oracle.seq_kv(w.seed, buf, b, L)
        qb = synth.q_rows(w.seed, synth.stream_q(layer), b, w.num_q_heads)
        o_ref, l_ref = oracle.decode_seq(qb, kc, ks, vc, vs, L, w.layer_windows[layer], w.softmax_scale)
        assert np.abs(out[b] - o_ref).max() <= ATOL, (layer, b)
        assert np.abs(lse[b] - l_ref).max() <= ATOL, (layer, b)


@pytest.mark.parametrize("P,W", [(16, 256), (32, 1024), (64, 100)])
def test_ring_decode_local(P, W):
    L = [W - 1, W, W + 1, 3 * W + 17, 5000, 777]
    w = synth.Workload("ring-decode", len(L), 32, P, np.asarray(L, dtype=np.int64), [W], [0], n_new=1, seed=41)
    cache = harness.PagedCache(w, local_ring=True)
    R = cai.cai_ring_pages(W, P, 1)
    assert cache.ring[0] == R and cache.pools[0].num_pages == w.batch * R
    cache.fill()
    cache.append_step()
    err, out, lse = decode_errs(cache, 0)
    assert err == 0
    check_decode(cache, 0, out, lse)


def test_ring_hybrid_layers_share_buffers():
    # Two local layers on a ringed buffer and one global layer on a full buffer.
    L = [200, 1500, 4097, 64]
    w = synth.Workload("ring-hybrid", len(L), 8, 16, np.asarray(L, dtype=np.int64), [512, 512, 0], [0, 0, 1],
                       n_new=1, seed=43)
    cache = harness.PagedCache(w, local_ring=True)
    assert cache.ring[0] > 0 and cache.ring[1] == 0
    cache.fill()
    cache.append_step()
    for layer in range(3):
        err, out, lse = decode_errs(cache, layer)
        assert err == 0
        check_decode(cache, layer, out, lse)


def test_ring_layers_one_launch():
    # The same three layers in one launch: ring tables for the local buffer, the full table for the global one.
    L = [200, 1500, 4097, 64]
    w = synth.Workload("ring-hybrid", len(L), 8, 16, np.asarray(L, dtype=np.int64), [512, 512, 0], [0, 0, 1],
                       n_new=1, seed=43)
    cache = harness.PagedCache(w, local_ring=True)
    cache.fill()
    cache.append_step()
    qs = [cache.decode_q(layer) for layer in range(3)]
    outs = [torch.full((w.batch, w.num_q_heads, 128), float("nan"), device="cuda") for _ in range(3)]
    lses = [torch.full((w.batch, w.num_q_heads), float("nan"), device="cuda") for _ in range(3)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.decode_layers(qs, outs, lses, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for layer in range(3):
        check_decode(cache, layer, outs[layer].cpu().numpy(), lses[layer].cpu().numpy())


def test_ring_prefill_window():
    W, n_new, P = 300, 64, 16
    L = np.asarray([2000, 64, 65 + W, 4001], dtype=np.int64)
    w = synth.Workload("ring-prefill", len(L), 32, P, L, [W], [0], n_new=n_new, seed=47)
    cache = harness.PagedCache(w, local_ring=True, ring_new_tokens=n_new)
    assert cache.ring[0] == cai.cai_ring_pages(W, P, n_new)
    cache.fill()
    cache.append_step()
    q = cache.prefill_q()
    out = torch.full((w.batch, n_new, 32, 128), float("nan"), device="cuda")
    lse = torch.full((w.batch, n_new, 32), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.prefill(q, out, lse, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(w.batch):
        Lb = int(L[b])
        kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, Lb)
        qb = synth.q_rows(w.seed, synth.STREAM_Q_PREFILL, b, n_new * 32).reshape(n_new, 32, 128)
        o_ref, l_ref = oracle.prefill_seq(qb, kc, ks, vc, vs, Lb - n_new, W, w.softmax_scale, None)
        assert np.abs(out[b] - o_ref).max() <= ATOL, b
        assert np.abs(lse[b] - l_ref).max() <= ATOL, b


def test_ring_one_page_short_is_caught():
    # With the ring one page shorter than needed, some decode must reach an entry
    # marked -1, and the kernel reports it instead of reading another position.
    W, P = 256, 16
    L = [W + 5, 3 * W + 9, 1000, 517]
    w = synth.Workload("ring-short", len(L), 8, P, np.asarray(L, dtype=np.int64), [W], [0], n_new=1, seed=53)
    cache = harness.PagedCache(w, local_ring=True)
    cache.fill()
    cache.append_step()
    R = cache.ring[0]
    short = np.stack([cai.cai_ring_table_row(cache.ring_ids[0][b][:R - 1], int(L[b]), P, cache.max_pages_per_seq)
                      for b in range(w.batch)])
    cache.ring_tables[0] = torch.from_numpy(short).to("cuda")
    err, _, _ = decode_errs(cache, 0)
    assert err & cai.CAI_DEVERR_PAGE

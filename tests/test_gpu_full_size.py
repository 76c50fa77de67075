"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic split plans, all layers of a step in one launch).

The split plan depends on the batch and the SM count, so a shrunk workload
does not exercise the plan that is benchmarked.  Here every workload runs at
its own size and a seeded sample of its sequences -- the shortest, the longest
and evenly spaced ones -- is compared element by element with the float64
oracle, within 2e-3 absolute:
  * the hybrid 6-layer step: batch 256, lognormal lengths, the step's appends
    into the four buffers, all six layers in one launch;
  * the long-context global decode: batch 1024, 64 heads, lengths up to
    131072 tokens, page size 64 (about 20 GB of KV);
  * the append-prefill chunk: batch 16, 8192-token prefixes, 256 new tokens,
    16 tokens per sampled sequence including the first and the last.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import harness  # noqa: E402
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


def sample(ctx_len, n):
    """Shortest, longest and n - 2 more evenly spaced by length (seeded ties by index)."""
    order = np.argsort(np.asarray(ctx_len), kind="stable")
    idx = np.linspace(0, len(order) - 1, n).round().astype(int)
    return list(dict.fromkeys(int(order[i]) for i in idx))


def check_decode_seqs(w, outs, lses, seqs, layers):
    """outs/lses: numpy per layer.  Returns the worst output error."""

    def one(b):
        L = int(w.ctx_len[b])
        kv = {}
        worst = 0.0
        for layer in layers:
            buf = w.layer_to_buffer[layer]
            if buf not in kv:
                kv[buf] = oracle.seq_kv(w.seed, buf, b, L)
            kc, ks, vc, vs = kv[buf]
            qb = synth.q_rows(w.seed, synth.stream_q(layer), b, w.num_q_heads)
            ref, ref_lse = oracle.decode_seq(qb, kc, ks, vc, vs, L, w.layer_windows[layer], w.softmax_scale)
            e = float(np.abs(outs[layer][b] - ref).max())
            assert e <= ATOL, (b, layer, e)
            assert np.abs(lses[layer][b] - ref_lse).max() <= ATOL, (b, layer)
            worst = max(worst, e)
        return worst

    with ThreadPoolExecutor(8) as ex:
        return max(ex.map(one, seqs))


def test_hybrid_step_full_size():
    w = synth.workload(3)
    assert w.batch == 256
    cache = harness.PagedCache(w)
    cache.fill()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.append_step(err=err)
    nl = len(w.layer_windows)
    qs = [cache.decode_q(layer) for layer in range(nl)]
    outs = [torch.full((w.batch, w.num_q_heads, 128), float("nan"), device="cuda") for _ in range(nl)]
    lses = [torch.full((w.batch, w.num_q_heads), float("nan"), device="cuda") for _ in range(nl)]
    cache.decode_layers(qs, outs, lses, err=err)  # automatic split plan, as benchmarked
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = [t.cpu().numpy() for t in outs]
    l = [t.cpu().numpy() for t in lses]
    assert all(np.isfinite(x).all() for x in o)
    seqs = sample(w.ctx_len, 10)
    assert len(seqs) >= 8
    check_decode_seqs(w, o, l, seqs, range(nl))


def test_long_global_full_size():
    w = synth.workload(5)
    assert w.batch == 1024 and w.num_q_heads == 64 and w.page_size == 64
    cache = harness.PagedCache(w)
    cache.fill()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.append_step(err=err)
    q = cache.decode_q(0)
    out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), device="cuda")
    lse = torch.full((w.batch, w.num_q_heads), float("nan"), device="cuda")
    cache.decode(0, q, out, lse, err=err)  # automatic split plan (8..32 splits at these lengths)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = out.cpu().numpy()
    assert np.isfinite(o).all()
    seqs = sample(w.ctx_len, 8)
    check_decode_seqs(w, [o], [lse.cpu().numpy()], seqs, [0])


def test_append_prefill_full_size():
    w = synth.workload(4)
    assert w.batch == 16 and w.n_new == 256
    cache = harness.PagedCache(w)
    cache.fill()
    k, v, start = cache.step_kv(0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    import int8_mqa_decode_gb300 as cai
    cai.cai_kv_append(cache.pools[0], k, v, cache.table, start, err_flag=err)
    q = cache.prefill_q()
    out = torch.full((w.batch, w.n_new, w.num_q_heads, 128), float("nan"), device="cuda")
    lse = torch.full((w.batch, w.n_new, w.num_q_heads), float("nan"), device="cuda")
    cache.prefill(q, out, lse, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(o).all()
    tokens = [0, 1, 2, 63, 64, 126, 127, 128, 129, 130, 191, 192, 200, 253, 254, 255]
    seqs = list(range(0, w.batch, 2))

    def one(b):
        L = int(w.ctx_len[b])
        kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, L)
        qb = synth.q_rows(w.seed, synth.STREAM_Q_PREFILL, b, w.n_new * w.num_q_heads).reshape(
            w.n_new, w.num_q_heads, 128)
        ref, ref_lse = oracle.prefill_seq(qb, kc, ks, vc, vs, L - w.n_new, 0, w.softmax_scale, tokens)
        e = float(np.abs(o[b][tokens] - ref).max())
        assert e <= ATOL, (b, e)
        assert np.abs(l[b][tokens] - ref_lse).max() <= ATOL, b
        return e

    with ThreadPoolExecutor(8) as ex:
        worst = max(ex.map(one, seqs))
    assert worst <= ATOL

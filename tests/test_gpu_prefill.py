"""GPU parity of the append-prefill attention against the oracle: causal
masks inside the chunk, windows, head counts, ragged q-tiles, the pages'
append-prefill workload shape (sampled tokens), and error handling."""
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


def prefill_case(B, Hq, P, prefix, n_new, window=0, seed=3):
    L = np.asarray(prefix, dtype=np.int64) + n_new
    w = synth.Workload("prefill-test", B, Hq, P, L, [window], [0], n_new=n_new, seed=seed)
    cache = harness.PagedCache(w)
    cache.fill()          # the reused prefix
    cache.append_step()   # the chunk's own K/V, quantized and appended first
    q = cache.prefill_q()
    out = torch.full((B, n_new, Hq, 128), float("nan"), device="cuda")
    lse = torch.full((B, n_new, Hq), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.prefill(q, out, lse, err=err)
    torch.cuda.synchronize()
    return w, cache, out.cpu().numpy(), lse.cpu().numpy(), int(err.item())


def oracle_prefill(w, b, tokens=None):
    L = int(w.ctx_len[b])
    kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, L)
    qb = synth.q_rows(w.seed, synth.STREAM_Q_PREFILL, b, w.n_new * w.num_q_heads).reshape(w.n_new, w.num_q_heads, 128)
    return oracle.prefill_seq(qb, kc, ks, vc, vs, L - w.n_new, w.layer_windows[0], w.softmax_scale, tokens)


def check(w, out, lse, tokens=None):
    for b in range(w.batch):
        o_ref, l_ref = oracle_prefill(w, b, tokens)
        sel = slice(None) if tokens is None else list(tokens)
        assert np.abs(out[b][sel] - o_ref).max() <= ATOL, b
        assert np.abs(lse[b][sel] - l_ref).max() <= ATOL, b


@pytest.mark.parametrize("Hq", [1, 8, 32, 128])
@pytest.mark.parametrize("prefix,n_new", [([0, 5], 1), ([0, 130], 3), ([127, 1], 9), ([300, 64], 40)])
def test_prefill_small_causal(Hq, prefix, n_new):
    w, cache, out, lse, err = prefill_case(2, Hq, 16, prefix, n_new)
    assert err == 0
    check(w, out, lse)


@pytest.mark.parametrize("P", [32, 64])
def test_prefill_page_sizes_and_window(P):
    w, cache, out, lse, err = prefill_case(2, 32, P, [3000, 700], 64, window=1024, seed=9)
    assert err == 0
    check(w, out, lse)


def test_prefill_workload_shape_sampled():
    # The append-prefill workload (prefix 8192, 256 new tokens, 32 heads) at batch 2, sampled tokens.
    w, cache, out, lse, err = prefill_case(2, 32, 16, [8192, 8192], 256, seed=1004)
    assert err == 0
    check(w, out, lse, tokens=[0, 1, 3, 4, 127, 128, 200, 255])


def test_prefill_last_token_matches_decode():
    w, cache, out, lse, err = prefill_case(3, 32, 16, [500, 1000, 77], 16, seed=21)
    q = cache.prefill_q()[:, -1].contiguous()  # the last new token's query, at position ctx_len - 1
    d_out = torch.empty(3, 32, 128, device="cuda")
    cai.cai_mqa_decode(cache.pools, [0], 0, q, cache.table, cache.ctx_len, 0, w.softmax_scale, 0,
                       cache.workspace(0), d_out)
    torch.cuda.synchronize()
    assert np.abs(out[:, -1] - d_out.cpu().numpy()).max() <= ATOL


def test_prefill_invalid_prefix_flags_and_zeroes():
    w, cache, out, lse, err = prefill_case(2, 8, 16, [40, 40], 8)
    prefix = torch.tensor([40, cache.max_pages_per_seq * 16], dtype=torch.int32, device="cuda")
    o = torch.full((2, 8, 8, 128), float("nan"), device="cuda")
    l = torch.full((2, 8, 8), float("nan"), device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    cai.cai_mqa_prefill_chunk(cache.pools[0], cache.prefill_q(), cache.table, prefix, 0, w.softmax_scale,
                              cache.prefill_workspace(), o, l, e)
    torch.cuda.synchronize()
    assert int(e.item()) == cai.CAI_DEVERR_LENGTH
    assert not o[1].cpu().numpy().any() and np.all(np.isneginf(l[1].cpu().numpy()))
    assert np.abs(o[0].cpu().numpy() - out[0]).max() == 0.0


@pytest.mark.parametrize("window", [0, 700])
def test_prefill_split_last_wave(window):
    """More q-tile pairs than SMs with a remainder: the pairs of the partial last wave are
    cut into key ranges and merged by their log-sum-exp.  Every token of the last sequence
    (whose pairs are the split ones) and a sample of the others, against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hq, n_new = 32, 256
    pairs_per_seq = n_new * Hq // 256
    B = sms // pairs_per_seq + 2          # a few pairs more than one wave
    assert (B * pairs_per_seq) % sms != 0
    prefix = [1500 + 37 * b for b in range(B)]
    w, cache, out, lse, err = prefill_case(B, Hq, 16, prefix, n_new, window=window, seed=9)
    assert err == 0
    assert np.isfinite(out).all()
    last = B - 1
    o_ref, l_ref = oracle_prefill(w, last)
    assert np.abs(out[last] - o_ref).max() <= ATOL
    assert np.abs(lse[last] - l_ref).max() <= ATOL
    tokens = [0, 1, 127, 128, 255]
    for b in (0, B // 2, B - 2):
        o_ref, l_ref = oracle_prefill(w, b, tokens)
        assert np.abs(out[b][tokens] - o_ref).max() <= ATOL, b
        assert np.abs(lse[b][tokens] - l_ref).max() <= ATOL, b


@pytest.mark.parametrize("q_scale", [8.0, 32.0])
def test_prefill_sharp_logits_raise_the_reference(q_scale):
    """Queries scaled by a power of two (exact in bf16): the half-row references rise many
    times along the keys and most weights underflow; sampled tokens against the oracle."""
    prefix, n_new = np.array([2500, 700]), 64
    w = synth.Workload("sharp-prefill", 2, 32, 16, prefix + n_new, [0], [0], n_new=n_new, seed=93)
    cache = harness.PagedCache(w)
    cache.fill()
    cache.append_step()
    q = cache.prefill_q().mul_(q_scale)
    out = torch.full((2, n_new, 32, 128), float("nan"), device="cuda")
    lse = torch.full((2, n_new, 32), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.prefill(q, out, lse, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got, got_lse = out.cpu().numpy(), lse.cpu().numpy()
    q_bits = q.view(torch.int16).cpu().numpy().view(np.uint16)
    tokens = [0, 1, 31, 62, 63]
    for b in range(2):
        L = int(w.ctx_len[b])
        kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, L)
        o_ref, l_ref = oracle.prefill_seq(q_bits[b], kc, ks, vc, vs, L - n_new, 0, w.softmax_scale, tokens)
        assert np.abs(got[b][tokens] - o_ref).max() <= ATOL, b
        assert np.abs(got_lse[b][tokens] - l_ref).max() <= ATOL, b

"""GPU parity of continuous batching: one launch over sequences that bring different
numbers of new tokens (one-token decode steps next to prefill chunks, an empty
sequence), packed by offsets, against the oracle's attention of each sequence; the
decode-step rows also against the decode path; invalid offsets are flagged and
leave the other sequences untouched."""
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


def mixed_case(prefix, n_new, Hq=32, P=16, window=0, seed=61, offsets=None):
    import synth.gpu as sgpu
    prefix = np.asarray(prefix, dtype=np.int64)
    n_new = np.asarray(n_new, dtype=np.int64)
    B = len(prefix)
    L = prefix + n_new
    w = synth.Workload("varlen", B, Hq, P, np.maximum(L, 1), [window], [0], n_new=1, seed=seed)
    cache = harness.PagedCache(w)
    cache.fill(upto=L)  # every sequence's prefix and its new tokens, appended
    off = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32) if offsets is None else np.asarray(offsets, np.int32)
    total = int(off[-1]) if offsets is None else int(n_new.sum())
    q = torch.zeros(max(total, 1), Hq, 128, dtype=torch.bfloat16, device="cuda")
    for b in range(B):
        if n_new[b] > 0 and offsets is None:
            qb = torch.empty(1, int(n_new[b]) * Hq, 128, dtype=torch.bfloat16, device="cuda")
            sgpu.q_rows(qb, w.seed, synth.STREAM_Q_PREFILL, b)
            q[off[b]:off[b + 1]] = qb.view(int(n_new[b]), Hq, 128)
    out = torch.full((max(total, 1), Hq, 128), float("nan"), device="cuda")
    lse = torch.full((max(total, 1), Hq), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = cache.prefill_workspace()
    cai.cai_mqa_prefill_varlen(cache.pools[0], q[:total] if total else q, torch.from_numpy(off).cuda(),
                               int(n_new.max()), cache.table, torch.from_numpy(prefix.astype(np.int32)).cuda(),
                               window, w.softmax_scale, ws, out[:total] if total else out,
                               lse[:total] if total else lse, err)
    torch.cuda.synchronize()
    return w, cache, off, out.cpu().numpy(), lse.cpu().numpy(), int(err.item())


def oracle_rows(w, b, p0, n, window):
    kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, p0 + n)
    qb = synth.q_rows(w.seed, synth.STREAM_Q_PREFILL, b, n * w.num_q_heads).reshape(n, w.num_q_heads, 128)
    return oracle.prefill_seq(qb, kc, ks, vc, vs, p0, window, w.softmax_scale, None)


@pytest.mark.parametrize("window", [0, 256])
def test_varlen_mixed_decode_and_prefill(window):
    prefix = [500, 4000, 300, 0, 1000, 77, 2047]
    n_new = [1, 1, 64, 3, 200, 0, 1]
    w, cache, off, out, lse, err = mixed_case(prefix, n_new, window=window)
    assert err == 0
    for b in range(len(prefix)):
        if n_new[b] == 0:
            continue
        o_ref, l_ref = oracle_rows(w, b, prefix[b], n_new[b], window)
        rows = slice(off[b], off[b + 1])
        assert np.abs(out[rows] - o_ref).max() <= ATOL, b
        assert np.abs(lse[rows] - l_ref).max() <= ATOL, b


def test_varlen_decode_rows_match_decode_path():
    import synth.gpu as sgpu
    prefix = [700, 3000, 64]
    n_new = [1, 1, 1]
    w, cache, off, out, lse, err = mixed_case(prefix, n_new, Hq=32, seed=67)
    assert err == 0
    # The decode path on the same cache (ctx_len = prefix + 1) with the same queries.
    q = torch.empty(3, 32, 128, dtype=torch.bfloat16, device="cuda")
    for b in range(3):
        qb = torch.empty(1, 32, 128, dtype=torch.bfloat16, device="cuda")
        sgpu.q_rows(qb, w.seed, synth.STREAM_Q_PREFILL, b)
        q[b] = qb[0]
    ctx = torch.tensor([p + 1 for p in prefix], dtype=torch.int32, device="cuda")
    d_out = torch.empty(3, 32, 128, device="cuda")
    ws = torch.zeros(cai.cai_mqa_decode_workspace_size(3, 32, cache.max_pages_per_seq, 16, 0, 0), dtype=torch.uint8,
                     device="cuda")
    cai.cai_mqa_decode(cache.pools, [0], 0, q, cache.table, ctx, 0, w.softmax_scale, 0, ws, d_out)
    torch.cuda.synchronize()
    assert np.abs(out[:3] - d_out.cpu().numpy()).max() <= ATOL


def test_varlen_invalid_offsets_flagged():
    # Sequence 2's end offset lies beyond the packed rows: flagged, nothing of it written,
    # and the rows of sequences 0 and 1 are still computed.
    prefix = [100, 200, 300]
    n_new = [4, 4, 4]
    offsets = [0, 4, 8, 100]
    w, cache, _, out, lse, err = mixed_case(prefix, n_new, offsets=offsets, seed=71)
    assert err & cai.CAI_DEVERR_LENGTH
    assert np.all(np.isfinite(out[0:8])) and np.all(np.isfinite(lse[0:8]))
    assert np.all(np.isnan(out[8:12])) and np.all(np.isnan(lse[8:12]))


def check_all_rows(w, off, out, lse, prefix, n_new, window=0):
    for b in range(len(prefix)):
        n = int(n_new[b])
        if n == 0:
            continue
        o_ref, l_ref = oracle_rows(w, b, int(prefix[b]), n, window)
        rows = slice(off[b], off[b + 1])
        assert np.abs(out[rows] - o_ref).max() <= ATOL, b
        assert np.abs(lse[rows] - l_ref).max() <= ATOL, b


@pytest.mark.parametrize("Hq,P", [(64, 16), (8, 32), (128, 64)])
def test_varlen_heads_and_page_sizes(Hq, P):
    """64 heads (the decode kernel's two-warpgroup softmax beside the prefill), a small
    head count with 32-token pages, and 128 heads (beyond the decode kernel: every row
    goes through the prefill kernel) with 64-token pages."""
    prefix = [900, 37, 2500, 400, 1]
    n_new = [1, 20, 1, 130, 1]
    w, cache, off, out, lse, err = mixed_case(prefix, n_new, Hq=Hq, P=P, seed=73)
    assert err == 0
    check_all_rows(w, off, out, lse, prefix, n_new)


def test_varlen_many_decode_rows_few_chunks():
    """Most of the batch is one-token rows: the decode launch beside the prefill's few
    q-tiles takes most of the SMs."""
    rng = np.random.default_rng(5)
    n_dec = 300
    prefix = np.concatenate([rng.integers(1, 3000, n_dec), [1500, 200]])
    n_new = np.concatenate([np.ones(n_dec, np.int64), [96, 33]])
    w, cache, off, out, lse, err = mixed_case(prefix, n_new, seed=79)
    assert err == 0
    sample = list(range(0, n_dec, 37)) + [n_dec - 1, n_dec, n_dec + 1]
    for b in sample:
        o_ref, l_ref = oracle_rows(w, b, int(prefix[b]), int(n_new[b]), 0)
        rows = slice(off[b], off[b + 1])
        assert np.abs(out[rows] - o_ref).max() <= ATOL, b
        assert np.abs(lse[rows] - l_ref).max() <= ATOL, b


def test_varlen_only_decode_rows():
    """No chunk at all: the prefill launch has no q-tile and the decode launch does everything."""
    prefix = [10, 1000, 5000, 129]
    n_new = [1, 1, 1, 1]
    w, cache, off, out, lse, err = mixed_case(prefix, n_new, seed=83)
    assert err == 0
    check_all_rows(w, off, out, lse, prefix, n_new)

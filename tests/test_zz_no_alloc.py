"""cai_mqa_decode_no_alloc, the decode entry point for callers that cannot
hand the library device scratch (allocation frozen after warm-up, plug-in
interfaces that pass only inputs and outputs, hosts whose framework owns all
device memory).  It must give what cai_mqa_decode gives, call after call,
while using only the scratch array built into the library."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = 2e-3


def test_no_alloc_matches_workspace_decode_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_mqa_decode_gb300 import build
    build.build()
    import harness
    import int8_mqa_decode_gb300 as cai
    import synth

    # The local-layer workload's shape at batch 16: 4 splits per sequence, so the scratch is really used.
    w = synth.workload(2, batch=16)
    cache = harness.PagedCache(w)
    cache.fill(upto=w.ctx_len)
    q = cache.decode_q(0)
    splits = 4
    assert 0 < cache.workspace(0, splits).numel() <= 32 << 20
    ref = torch.empty(w.batch, w.num_q_heads, 128, device="cuda")
    ref_lse = torch.empty(w.batch, w.num_q_heads, device="cuda")
    cache.decode(0, q, ref, ref_lse, num_splits=splits)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        cai.cai_mqa_decode_no_alloc(cache.pools, w.layer_to_buffer, 0, q, cache.table, cache.ctx_len,
                                    w.layer_windows[0], w.softmax_scale, splits, out, lse, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert np.abs(out.cpu().numpy() - ref.cpu().numpy()).max() <= ATOL
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= ATOL
    # ... and what the oracle gives, sequence by sequence.
    import oracle
    got, got_lse = out.cpu().numpy(), lse.cpu().numpy()
    qb_all = q.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(w.batch):
        L = int(w.ctx_len[b])
        kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, L)
        o_ref, l_ref = oracle.decode_seq(qb_all[b], kc, ks, vc, vs, L, w.layer_windows[0], w.softmax_scale)
        assert np.abs(got[b] - o_ref).max() <= ATOL, b
        assert np.abs(got_lse[b] - l_ref).max() <= ATOL, b
    # A plan that needs more scratch than the built-in array is refused before any launch.
    need = cai.cai_mqa_decode_workspace_size(64, 64, 2048, 64, 0, 64)
    assert need > 32 << 20
    with pytest.raises(cai.CaiError) as e:
        cai.cai_mqa_decode_no_alloc(cache.pools, [0], 0, torch.zeros(64, 64, 128, dtype=torch.bfloat16, device="cuda"),
                                    torch.zeros(64, 2048, dtype=torch.int32, device="cuda"),
                                    torch.zeros(64, dtype=torch.int32, device="cuda"), 0, 0.088, 64,
                                    torch.empty(64, 64, 128, device="cuda"))
    assert e.value.status == 3

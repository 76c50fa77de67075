"""Failure detection inside the kernels: every wait is bounded, and a wait that runs
out makes the launch report CAI_DEVERR_TIMEOUT, stop, wait for its own copies and
MMAs in flight and return, leaving the GPU usable.  The failure is made on the host:
with the fault injection on, every CTA skips the load of one of its K/V stages (a
message that never comes), and with a 20 ms wait limit the waits for it run out.
Ordinary calls afterwards must match the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import harness  # noqa: E402
import int8_mqa_decode_gb300 as cai  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

ATOL = 2e-3
LIMIT_NS = 20_000_000


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_mqa_decode_gb300 import build
    build.build()
    yield
    cai.cai_set_fault_injection(-1)
    cai.cai_set_wait_limit_ns(0)


def timed_out(call, stage):
    """Run call(err) with stage `stage` of every CTA dropped; True if the launch reported the timeout."""
    cai.cai_set_wait_limit_ns(LIMIT_NS)
    cai.cai_set_fault_injection(stage)
    try:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        call(err)
        torch.cuda.synchronize()
        return bool(int(err.item()) & cai.CAI_DEVERR_TIMEOUT)
    finally:
        cai.cai_set_fault_injection(-1)
        cai.cai_set_wait_limit_ns(0)


def test_decode_gives_up_then_recovers():
    w = synth.Workload("timeout-decode", 6, 32, 16, np.array([300, 2000, 5000, 64, 1500, 900]), [0], [0], seed=31)
    cache = harness.PagedCache(w)
    cache.fill(upto=w.ctx_len)
    q = cache.decode_q(0)
    out = torch.empty(w.batch, w.num_q_heads, 128, device="cuda")
    lse = torch.empty(w.batch, w.num_q_heads, device="cuda")
    ws = cache.workspace(0, 4)
    assert timed_out(lambda err: cache.decode(0, q, out, lse, num_splits=4, workspace=ws, err=err), 3)
    # Same workspace, default limit: the launch that gave up left the queue counters
    # at zero (every CTA's scheduler still counts itself out), so nothing is reset here.
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    cache.decode(0, q, out, lse, num_splits=4, workspace=ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got, got_lse = out.cpu().numpy(), lse.cpu().numpy()
    q_bits = q.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(w.batch):
        L = int(w.ctx_len[b])
        kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, L)
        o_ref, l_ref = oracle.decode_seq(q_bits[b], kc, ks, vc, vs, L, 0, w.softmax_scale)
        assert np.abs(got[b] - o_ref).max() <= ATOL, b
        assert np.abs(got_lse[b] - l_ref).max() <= ATOL, b


def test_decode_layers_gives_up_then_recovers():
    """The one-launch multi-layer step (64 heads: the two-warpgroup softmax)."""
    w = synth.Workload("timeout-layers", 3, 64, 64, np.array([4000, 130, 9000]), [0, 512], [0, 0], seed=34)
    cache = harness.PagedCache(w)
    cache.fill(upto=w.ctx_len)
    qs = [cache.decode_q(l) for l in range(2)]
    outs = [torch.empty(w.batch, w.num_q_heads, 128, device="cuda") for _ in range(2)]
    ws = cache.layers_workspace(0)
    assert timed_out(lambda err: cache.decode_layers(qs, outs, workspace=ws, err=err), 2)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for o in outs:
        o.fill_(float("nan"))
    cache.decode_layers(qs, outs, workspace=ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(2):
        got = outs[l].cpu().numpy()
        q_bits = qs[l].view(torch.int16).cpu().numpy().view(np.uint16)
        for b in range(w.batch):
            L = int(w.ctx_len[b])
            kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, L)
            o_ref, _ = oracle.decode_seq(q_bits[b], kc, ks, vc, vs, L, w.layer_windows[l], w.softmax_scale)
            assert np.abs(got[b] - o_ref).max() <= ATOL, (l, b)


def test_prefill_gives_up_then_recovers():
    prefix, n_new = np.array([700, 1300]), 64
    w = synth.Workload("timeout-prefill", 2, 32, 16, prefix + n_new, [0], [0], n_new=n_new, seed=33)
    cache = harness.PagedCache(w)
    cache.fill()
    cache.append_step()
    q = cache.prefill_q()
    out = torch.empty(w.batch, n_new, w.num_q_heads, 128, device="cuda")
    lse = torch.empty(w.batch, n_new, w.num_q_heads, device="cuda")
    ws = cache.prefill_workspace()
    assert timed_out(lambda err: cache.prefill(q, out, lse, workspace=ws, err=err), 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    cache.prefill(q, out, lse, workspace=ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got, got_lse = out.cpu().numpy(), lse.cpu().numpy()
    tokens = [0, 31, 63]
    for b in range(w.batch):
        L = int(w.ctx_len[b])
        kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, L)
        qb = synth.q_rows(w.seed, synth.STREAM_Q_PREFILL, b, n_new * w.num_q_heads).reshape(n_new, w.num_q_heads, 128)
        o_ref, l_ref = oracle.prefill_seq(qb, kc, ks, vc, vs, L - n_new, 0, w.softmax_scale, tokens)
        assert np.abs(got[b][tokens] - o_ref).max() <= ATOL, b
        assert np.abs(got_lse[b][tokens] - l_ref).max() <= ATOL, b


def test_varlen_gives_up_then_recovers():
    """A continuous-batching call: its prefill launch and the decode launch that runs beside it
    (without waiting for it) both give up; the call still ends, and the next one is right."""
    import synth.gpu as sgpu
    synth.gpu.build()
    prefix = np.array([900, 3000, 500, 2000, 64])
    n_new = np.array([1, 128, 1, 64, 1])
    L = prefix + n_new
    w = synth.Workload("timeout-varlen", len(prefix), 32, 16, L, [0], [0], n_new=1, seed=36)
    cache = harness.PagedCache(w)
    cache.fill(upto=L)
    off = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    total = int(off[-1])
    q = torch.empty(total, w.num_q_heads, 128, dtype=torch.bfloat16, device="cuda")
    for b in range(len(prefix)):
        qb = torch.empty(1, int(n_new[b]) * w.num_q_heads, 128, dtype=torch.bfloat16, device="cuda")
        sgpu.q_rows(qb, w.seed, synth.STREAM_Q_PREFILL, b)
        q[off[b]:off[b + 1]] = qb.view(int(n_new[b]), w.num_q_heads, 128)
    off_d = torch.from_numpy(off).cuda()
    prefix_d = torch.from_numpy(prefix.astype(np.int32)).cuda()
    out = torch.empty(total, w.num_q_heads, 128, device="cuda")
    lse = torch.empty(total, w.num_q_heads, device="cuda")
    ws = cache.prefill_workspace()

    def call(err):
        cai.cai_mqa_prefill_varlen(cache.pools[0], q, off_d, int(n_new.max()), cache.table, prefix_d, 0,
                                   w.softmax_scale, ws, out, lse, err)

    assert timed_out(call, 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    call(err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got, got_lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(len(prefix)):
        n = int(n_new[b])
        kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, int(L[b]))
        qb = synth.q_rows(w.seed, synth.STREAM_Q_PREFILL, b, n * w.num_q_heads).reshape(n, w.num_q_heads, 128)
        tokens = [0, n - 1] if n > 1 else [0]
        o_ref, l_ref = oracle.prefill_seq(qb, kc, ks, vc, vs, int(prefix[b]), 0, w.softmax_scale, tokens)
        rows = [int(off[b]) + t for t in tokens]
        assert np.abs(got[rows] - o_ref).max() <= ATOL, b
        assert np.abs(got_lse[rows] - l_ref).max() <= ATOL, b


def test_defaults_are_restored():
    """After the tests above the injection is off and the default limit is back."""
    w = synth.workload(1)
    cache = harness.PagedCache(w)
    cache.fill(upto=w.ctx_len)
    q = cache.decode_q(0)
    out = torch.empty(w.batch, w.num_q_heads, 128, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache.decode(0, q, out, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

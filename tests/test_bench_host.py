"""Host-side logic of bench.py: work accounting and the multi-rank plumbing
(gloo, world size 2, CPU only)."""
import os
import socket

import numpy as np
import pytest

import bench
import synth


def test_layer_work_counts_attended_tokens_and_pages_by_brute_force():
    w = synth.workload(3, batch=40)
    for layer in (0, 5):
        toks, pages, byts = bench.layer_work(w, layer)
        W = w.layer_windows[layer]
        bt, bp = 0, 0
        for L in w.ctx_len:
            pos = [p for p in range(int(L)) if (W == 0 or p >= L - W)]
            bt += len(pos)
            bp += len({p // w.page_size for p in pos})
        assert toks == bt and pages == bp
        assert byts == bt * 264 + bp * 4 + w.batch * w.num_q_heads * 128 * 6 + w.batch * 4


def test_step_work_sums_layers():
    w = synth.workload(3)
    toks, _ = bench.step_work(w)
    L = np.asarray(w.ctx_len)
    assert toks == int((5 * np.minimum(L, 1024) + L).sum())


def test_l2_flush_only_for_workloads_that_fit_twice_in_l2():
    # The decode bench flushes L2 between timed steps exactly when a step's KV bytes are
    # below twice the L2: the tiny and the local-layer workloads, not the hybrid step or
    # the long-context one (which read more than the L2 holds every step).
    flushed = {n: bench.step_work(synth.workload(n))[1] < 2 * bench.L2_BYTES for n in (1, 2, 3, 5)}
    assert flushed == {1: True, 2: True, 3: False, 5: False}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, wsz = bench.dist_init()
    bench.barrier(wsz)
    m = bench.allreduce_max(10.0 + rank, wsz)
    # Each rank's batch is independent: different seeds, same shapes (weak scaling).
    w = synth.workload(3, seed=1003 + 100 * r, batch=8)
    q.put((r, wsz, m, int(w.ctx_len.sum())))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_gloo_max_and_weak_sharding():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[2] == 11.0 for r in res)       # max over ranks
    assert res[0][3] != res[1][3]               # different data per rank

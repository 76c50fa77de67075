"""The GPU generator gives the same bits as the numpy one."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402


def test_gpu_generator_matches_numpy():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import synth.gpu as sg
    out = torch.empty(3, 50, 128, dtype=torch.float32, device="cuda")
    pos = torch.tensor([0, 1000, 123456], dtype=torch.int32, device="cuda")
    sg.normal_rows(out, 99, synth.stream_v(2), 7, pos=pos)
    got = out.cpu().numpy()
    for i, p in enumerate([0, 1000, 123456]):
        assert np.array_equal(got[i], synth.kv_rows(99, synth.stream_v(2), 7 + i, p, 50))
    q = torch.empty(2, 64, 128, dtype=torch.bfloat16, device="cuda")
    sg.q_rows(q, 99, synth.stream_q(3), 5)
    qb = q.view(torch.int16).cpu().numpy().view(np.uint16)
    for i in range(2):
        assert np.array_equal(qb[i], synth.q_rows(99, synth.stream_q(3), 5 + i, 64))

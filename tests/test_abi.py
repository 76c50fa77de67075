"""The C ABI without a GPU: the library loads, exports every function the
header declares, and its host-side validation answers with status codes
before any launch."""
import ctypes
import os
import re

import pytest

import int8_mqa_decode_gb300 as cai
from int8_mqa_decode_gb300 import build as cai_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails before any launch


@pytest.fixture(scope="module")
def lib():
    cai_build.build()
    return cai.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "cai.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cai_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"cai_kv_append", "cai_mqa_decode", "cai_mqa_prefill_chunk", "cai_mqa_decode_workspace_size",
            "cai_status_string", "cai_page_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_page_bytes_and_status_strings(lib):
    assert cai.cai_page_bytes(16) == 16 * 264 == 4224
    assert cai.cai_page_bytes(64) == 16896
    assert cai.cai_page_bytes(0) == 0
    assert cai.cai_status_string(0) == "ok"
    assert "workspace" in cai.cai_status_string(3)


def test_workspace_size_plan(lib):
    # One split needs only the 256-byte work-queue header; a 1024-position window in 4 splits also
    # needs [B][4][Hq] partial outputs and log-sum-exps.
    assert cai.cai_mqa_decode_workspace_size(4, 8, 32, 16, 0, 1) == 256
    ws = cai.cai_mqa_decode_workspace_size(256, 32, 2048, 16, 1024, 4)
    rows = 256 * 4 * 32
    assert ws == 256 + ((rows * 128 * 4 + 255) // 256) * 256 + ((rows * 4 + 255) // 256) * 256
    assert cai.cai_mqa_decode_workspace_size(4, 8, 32, 24, 0, 0) == 0  # unsupported page size
    assert cai.cai_mqa_decode_workspace_size(4, 8, 32, 16, 0, 65) == 0  # too many splits


def _pool(num_pages=8, page_size=16, head_dim=128, pages=FAKE):
    return cai.cai_kv_pool(pages, num_pages, page_size, head_dim)


def test_append_validation(lib):
    pool = _pool()
    ok_args = dict(k=FAKE, v=FAKE, batch=2, n_new=1, table=FAKE, maxp=4, start=FAKE)

    def call(pool, **kw):
        a = dict(ok_args, **kw)
        return lib.cai_kv_append(ctypes.byref(pool), a["k"], a["v"], a["batch"], a["n_new"], a["table"], a["maxp"],
                                 a["start"], None, None)

    assert lib.cai_kv_append(None, FAKE, FAKE, 1, 1, FAKE, 4, FAKE, None, None) == 1
    assert call(_pool(head_dim=64)) == 2
    assert call(_pool(page_size=24)) == 2
    assert call(_pool(page_size=128)) == 2
    assert call(_pool(pages=FAKE + 4)) == 1     # misaligned pool
    assert call(pool, k=FAKE + 8) == 1          # misaligned input
    assert call(pool, table=None) == 1
    assert call(pool, batch=-1) == 1
    assert call(pool, batch=0) == 0             # nothing to do, nothing launched
    assert call(pool, n_new=0) == 0


def test_append_pools_validation(lib):
    pools = (cai.cai_kv_pool * 2)(_pool(), _pool())
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)

    def call(pools=pools, n=2, k=arr, v=arr, batch=2, n_new=1, tables=arr, maxp=4, start=arr):
        return lib.cai_kv_append_pools(pools, n, k, v, batch, n_new, tables, maxp, start, None, None)

    assert call(n=0) == 2
    assert call(n=9) == 2
    assert call(k=None) == 1
    assert call(v=(ctypes.c_void_p * 2)(FAKE, FAKE + 4)) == 1  # misaligned
    assert call(start=(ctypes.c_void_p * 2)(FAKE, None)) == 1
    assert call(maxp=0) == 1
    assert call(pools=(cai.cai_kv_pool * 2)(_pool(), _pool(head_dim=96))) == 2
    assert call(batch=0) == 0


def test_decode_validation(lib):
    pools = (cai.cai_kv_pool * 2)(_pool(), _pool())
    l2p = (ctypes.c_int32 * 3)(0, 0, 1)

    def call(**kw):
        a = dict(pools=pools, npools=2, l2p=l2p, nlayers=3, layer=0, q=FAKE, batch=2, hq=8, table=FAKE, maxp=64,
                 ctx=FAKE, window=0, scale=0.088, splits=1, ws=None, ws_bytes=0, out=FAKE)
        a.update(kw)
        return lib.cai_mqa_decode(a["pools"], a["npools"], a["l2p"], a["nlayers"], a["layer"], a["q"], a["batch"],
                                  a["hq"], a["table"], a["maxp"], a["ctx"], a["window"], a["scale"], a["splits"],
                                  a["ws"], a["ws_bytes"], a["out"], None, None, None)

    assert call(layer=3) == 1
    assert call(layer=2, l2p=(ctypes.c_int32 * 3)(0, 0, 2)) == 1  # buffer index out of range
    assert call(hq=0) == 2
    assert call(hq=65) == 2
    assert call(q=FAKE + 2) == 1
    assert call(out=None) == 1
    assert call(window=-1) == 1
    assert call(splits=65) == 1
    assert call(scale=float("nan")) == 1
    assert call(batch=0) == 0
    # Every decode needs a workspace (at least its 256-byte header); every call here fails before any launch.
    assert call(splits=1) == 3
    assert call(splits=4, ws=FAKE, ws_bytes=16) == 3
    assert call(splits=1, ws=FAKE + 16, ws_bytes=4096) == 3  # not 256-byte aligned
    bad = (cai.cai_kv_pool * 1)(_pool(head_dim=96))
    assert call(pools=bad, npools=1, l2p=(ctypes.c_int32 * 1)(0), nlayers=1) == 2


def test_decode_layers_validation(lib):
    pools = (cai.cai_kv_pool * 2)(_pool(), _pool())

    def arr(ctype, vals):
        return (ctype * len(vals))(*vals)

    def call(n=3, **kw):
        a = dict(pools=pools, npools=2, l2p=arr(ctypes.c_int32, [0, 0, 1][:n] + [0] * max(0, n - 3)),
                 windows=arr(ctypes.c_int32, [1024, 1024, 0][:n] + [0] * max(0, n - 3)),
                 q=arr(ctypes.c_void_p, [FAKE] * n), batch=2, hq=8, tables=arr(ctypes.c_void_p, [FAKE] * n),
                 maxp=64, ctx=FAKE, scale=0.088, splits=0, ws=None, ws_bytes=0,
                 out=arr(ctypes.c_void_p, [FAKE] * n))
        a.update(kw)
        return lib.cai_mqa_decode_layers(a["pools"], a["npools"], a["l2p"], n, a["windows"], a["q"], a["batch"],
                                         a["hq"], a["tables"], a["maxp"], a["ctx"], a["scale"], a["splits"], a["ws"],
                                         a["ws_bytes"], a["out"], None, None, None)

    assert call(n=0) == 2
    assert call(n=9) == 2
    assert call(l2p=arr(ctypes.c_int32, [0, 0, 2])) == 1  # buffer index out of range
    assert call(windows=arr(ctypes.c_int32, [1024, -1, 0])) == 1
    assert call(q=arr(ctypes.c_void_p, [FAKE, FAKE + 4, FAKE])) == 1
    assert call(out=arr(ctypes.c_void_p, [FAKE, None, FAKE])) == 1
    assert call(tables=None) == 1
    assert call(hq=65) == 2
    assert call(scale=float("nan")) == 1
    assert call(batch=0) == 0
    assert call() == 3  # no workspace
    assert call(ws=FAKE, ws_bytes=16) == 3
    mixed = (cai.cai_kv_pool * 2)(_pool(), _pool(page_size=32))
    assert call(pools=mixed) == 1  # one page size per call
    windows = arr(ctypes.c_int32, [1024, 0])
    one = lib.cai_mqa_decode_workspace_size(2, 8, 64, 16, 0, 0)
    both = lib.cai_mqa_decode_layers_workspace_size(2, 8, 64, 16, 2, windows, 0)
    assert both >= one and lib.cai_mqa_decode_layers_workspace_size(2, 8, 64, 16, 9, windows, 0) == 0


def test_prefill_varlen_validation(lib):
    pool = _pool()

    def call(**kw):
        a = dict(q=FAKE, batch=3, off=FAKE, total=40, maxn=32, hq=8, table=FAKE, maxp=64, prefix=FAKE, window=0,
                 scale=0.088, ws=None, ws_bytes=0, out=FAKE)
        a.update(kw)
        return lib.cai_mqa_prefill_varlen(ctypes.byref(pool), a["q"], a["batch"], a["off"], a["total"], a["maxn"],
                                          a["hq"], a["table"], a["maxp"], a["prefix"], a["window"], a["scale"],
                                          a["ws"], a["ws_bytes"], a["out"], None, None, None)

    assert call(off=None) == 1          # offsets are required
    assert call(hq=6) == 2              # heads a power of two
    assert call(hq=256) == 2
    assert call(total=-1) == 1
    assert call(maxn=-1) == 1
    assert call(window=-1) == 1
    assert call(q=FAKE + 4) == 1
    assert call(out=None) == 1
    assert call(batch=0) == 0           # nothing to do, nothing launched
    assert call(total=0) == 0
    assert call(maxn=0) == 0
    assert call() == 3                  # every call here stops at the workspace check
    assert call(ws=FAKE + 16, ws_bytes=1 << 30) == 3


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    pool = cai.KVPool.__new__(cai.KVPool)
    pool.struct = _pool()
    pool.head_dim = 128
    x = torch.zeros(1, 1, 128)
    with pytest.raises(ValueError):
        cai.cai_kv_append(pool, x, x, torch.zeros(1, 4, dtype=torch.int32), torch.zeros(1, dtype=torch.int32))

"""Python binding of libcai, the int8 MQA paged-KV decode library (include/cai.h).

Argument marshalling only: each function checks tensor devices, dtypes,
shapes and contiguity, turns them into pointers and sizes, and calls the C
entry point of the same name on the current CUDA stream.  Every step of the
computation runs in the CUDA kernels behind libcai.so; there is no CPU or
eager fallback.  If the compiled library is missing, importing the binding's
functions raises ``CaiUnavailable``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

__all__ = [
    "CaiError", "CaiUnavailable", "KVPool", "library_path", "load", "cai_page_bytes", "cai_status_string",
    "cai_kv_append", "cai_kv_append_pools", "cai_mqa_decode_workspace_size", "cai_mqa_decode", "cai_mqa_decode_no_alloc",
    "cai_mqa_decode_layers_workspace_size", "cai_mqa_decode_layers",
    "cai_mqa_prefill_workspace_size",
    "cai_mqa_prefill_chunk", "cai_mqa_prefill_varlen", "cai_gqa_decode", "cai_gqa_decode_workspace_size",
    "CAI_DEVERR_PAGE", "CAI_DEVERR_LENGTH", "CAI_DEVERR_TIMEOUT", "HEAD_DIM", "cai_host_cache_create",
    "cai_host_cache_destroy", "cai_host_cache_match", "cai_host_cache_restore", "cai_host_cache_store",
    "cai_host_cache_stats", "cai_host_cache_restore_batch", "cai_set_wait_limit_ns", "cai_set_fault_injection", "cai_ring_pages", "cai_ring_table_row",
]

HEAD_DIM = 128
CAI_OK, CAI_ERR_INVALID_ARG, CAI_ERR_UNSUPPORTED, CAI_ERR_WORKSPACE, CAI_ERR_CUDA = range(5)
CAI_DEVERR_PAGE, CAI_DEVERR_LENGTH, CAI_DEVERR_TIMEOUT = 1, 2, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


class CaiUnavailable(RuntimeError):
    """The compiled CUDA library (libcai.so) is not there or does not load."""


class CaiError(RuntimeError):
    def __init__(self, status: int, where: str):
        detail = f": {load().cai_last_cuda_error().decode()}" if status == CAI_ERR_CUDA else ""
        super().__init__(f"{where}: {cai_status_string(status)} (status {status}){detail}")
        self.status = status


class cai_kv_pool(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


def library_path() -> str:
    return os.path.join(_HERE, "libcai.so")


def load():
    """Load libcai.so (built by ``build.py``); raise CaiUnavailable if it cannot be loaded."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise CaiUnavailable(f"{path} is missing: build it with `python -m int8_mqa_decode_gb300.build`")
    try:
        lib = ctypes.CDLL(path)
    except OSError as e:  # pragma: no cover - depends on the machine
        raise CaiUnavailable(f"cannot load {path}: {e}") from e
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    pool_p = ctypes.POINTER(cai_kv_pool)
    lib.cai_page_bytes.argtypes = [i32, i32]
    lib.cai_page_bytes.restype = sz
    lib.cai_status_string.argtypes = [ctypes.c_int]
    lib.cai_status_string.restype = ctypes.c_char_p
    lib.cai_last_cuda_error.argtypes = []
    lib.cai_last_cuda_error.restype = ctypes.c_char_p
    lib.cai_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.cai_set_wait_limit_ns.restype = None
    lib.cai_set_fault_injection.argtypes = [ctypes.c_int32]
    lib.cai_set_fault_injection.restype = None
    lib.cai_kv_append.argtypes = [pool_p, vp, vp, i32, i32, vp, i32, vp, vp, vp]
    lib.cai_kv_append.restype = ctypes.c_int
    lib.cai_kv_append_pools.argtypes = [pool_p, i32, vp, vp, i32, i32, vp, i32, vp, vp, vp]
    lib.cai_kv_append_pools.restype = ctypes.c_int
    lib.cai_mqa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.cai_mqa_decode_workspace_size.restype = sz
    lib.cai_mqa_decode.argtypes = [pool_p, i32, vp, i32, i32, vp, i32, i32, vp, i32, vp, i32, ctypes.c_float, i32,
                                   vp, sz, vp, vp, vp, vp]
    lib.cai_mqa_decode.restype = ctypes.c_int
    lib.cai_mqa_decode_no_alloc.argtypes = [pool_p, i32, vp, i32, i32, vp, i32, i32, vp, i32, vp, i32,
                                            ctypes.c_float, i32, vp, vp, vp, vp]
    lib.cai_mqa_decode_no_alloc.restype = ctypes.c_int
    lib.cai_mqa_prefill_workspace_size.argtypes = [i32, i32, i32]
    lib.cai_mqa_prefill_workspace_size.restype = sz
    lib.cai_mqa_prefill_chunk.argtypes = [pool_p, vp, i32, i32, i32, vp, i32, vp, i32, ctypes.c_float, vp, sz, vp, vp,
                                          vp, vp]
    lib.cai_mqa_prefill_chunk.restype = ctypes.c_int
    lib.cai_mqa_prefill_varlen.argtypes = [pool_p, vp, i32, vp, i32, i32, i32, vp, i32, vp, i32, ctypes.c_float, vp,
                                           sz, vp, vp, vp, vp]
    lib.cai_mqa_prefill_varlen.restype = ctypes.c_int
    lib.cai_mqa_decode_layers_workspace_size.argtypes = [i32, i32, i32, i32, i32, vp, i32]
    lib.cai_mqa_decode_layers_workspace_size.restype = sz
    lib.cai_mqa_decode_layers.argtypes = [pool_p, i32, vp, i32, vp, vp, i32, i32, vp, i32, vp, ctypes.c_float, i32,
                                          vp, sz, vp, vp, vp, vp]
    lib.cai_mqa_decode_layers.restype = ctypes.c_int
    lib.cai_gqa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.cai_gqa_decode_workspace_size.restype = sz
    lib.cai_gqa_decode.argtypes = [pool_p, i32, vp, i32, i32, vp, i32, vp, i32, ctypes.c_float, i32, vp, sz, vp, vp,
                                   vp, vp]
    lib.cai_gqa_decode.restype = ctypes.c_int
    lib.cai_host_cache_create.argtypes = [i32, i32, i32, ctypes.c_int64]
    lib.cai_host_cache_create.restype = vp
    lib.cai_host_cache_destroy.argtypes = [vp]
    lib.cai_host_cache_destroy.restype = None
    lib.cai_host_cache_match.argtypes = [vp, vp, i32]
    lib.cai_host_cache_match.restype = i32
    lib.cai_host_cache_restore.argtypes = [vp, vp, i32, pool_p, vp, vp]
    lib.cai_host_cache_restore.restype = ctypes.c_int
    lib.cai_host_cache_restore_batch.argtypes = [vp, i32, vp, vp, pool_p, vp, vp]
    lib.cai_host_cache_restore_batch.restype = ctypes.c_int
    lib.cai_host_cache_store.argtypes = [vp, vp, i32, pool_p, vp, vp]
    lib.cai_host_cache_store.restype = ctypes.c_int
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.cai_host_cache_stats.argtypes = [vp, i64p, i64p, i64p, i64p]
    lib.cai_host_cache_stats.restype = None
    lib.cai_ring_pages.argtypes = [i32, i32, i32]
    lib.cai_ring_pages.restype = i32
    lib.cai_ring_table_row.argtypes = [vp, i32, vp, i32, i32, i32]
    lib.cai_ring_table_row.restype = ctypes.c_int
    _lib = lib
    return lib


def cai_status_string(status: int) -> str:
    return load().cai_status_string(int(status)).decode()


def cai_page_bytes(page_size: int, head_dim: int = HEAD_DIM) -> int:
    return int(load().cai_page_bytes(page_size, head_dim))


def _check(status: int, where: str) -> None:
    if status != CAI_OK:
        raise CaiError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, shape=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


class KVPool:
    """One KV buffer: ``num_pages`` pages of ``page_size`` tokens in one uint8 CUDA tensor.

    Page layout: K codes int8 [P][128], V codes int8 [P][128], K scales fp32 [P],
    V scales fp32 [P].  ``pages`` may also be given (any uint8 CUDA tensor of the
    right size, e.g. a view into a larger arena).
    """

    def __init__(self, num_pages: int, page_size: int, head_dim: int = HEAD_DIM, device=None,
                 pages: Optional[torch.Tensor] = None):
        nbytes = num_pages * cai_page_bytes(page_size, head_dim)
        if pages is None:
            pages = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
        if pages.dtype != torch.uint8 or pages.numel() != nbytes or not pages.is_cuda:
            raise ValueError("pages must be a uint8 CUDA tensor of num_pages * page_bytes bytes")
        self.pages = pages
        self.num_pages, self.page_size, self.head_dim = num_pages, page_size, head_dim
        self.struct = cai_kv_pool(pages.data_ptr(), num_pages, page_size, head_dim)


def cai_kv_append(pool: KVPool, k_new: torch.Tensor, v_new: torch.Tensor, block_table: torch.Tensor,
                  start_pos: torch.Tensor, err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """Quantize k_new/v_new fp32 [batch][n_new][128] to int8 and write them at start_pos[b] + i."""
    batch, n_new = (k_new.shape[0], k_new.shape[1]) if k_new.dim() == 3 else (0, 0)
    shape = (batch, n_new, pool.head_dim)
    st = load().cai_kv_append(
        ctypes.byref(pool.struct), _ptr(k_new, "k_new", torch.float32, shape), _ptr(v_new, "v_new", torch.float32, shape),
        batch, n_new, _ptr(block_table, "block_table", torch.int32), block_table.shape[-1],
        _ptr(start_pos, "start_pos", torch.int32, (batch,)), _ptr(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "cai_kv_append")


def cai_kv_append_pools(pools: Sequence[KVPool], k_new: Sequence[torch.Tensor], v_new: Sequence[torch.Tensor],
                        block_tables: Sequence[torch.Tensor], start_pos: Sequence[torch.Tensor],
                        err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """cai_kv_append into every pool of the list in one launch (entry i of each list goes to pools[i])."""
    n = len(pools)
    if not (len(k_new) == len(v_new) == len(block_tables) == len(start_pos) == n):
        raise ValueError("k_new, v_new, block_tables and start_pos must have one entry per pool")
    batch, n_new = (k_new[0].shape[0], k_new[0].shape[1]) if k_new[0].dim() == 3 else (0, 0)
    max_pages = block_tables[0].shape[-1]
    for t in block_tables:
        if t.shape[-1] != max_pages:
            raise ValueError("block tables of one call must have the same width")
    shape = (batch, n_new, HEAD_DIM)
    ks = (ctypes.c_void_p * n)(*[_ptr(t, "k_new", torch.float32, shape) for t in k_new])
    vs = (ctypes.c_void_p * n)(*[_ptr(t, "v_new", torch.float32, shape) for t in v_new])
    ts = (ctypes.c_void_p * n)(*[_ptr(t, "block_table", torch.int32) for t in block_tables])
    ss = (ctypes.c_void_p * n)(*[_ptr(t, "start_pos", torch.int32, (batch,)) for t in start_pos])
    st = load().cai_kv_append_pools(_pool_array(pools), n, ks, vs, batch, n_new, ts, max_pages, ss,
                                    _ptr(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "cai_kv_append_pools")


def cai_mqa_decode_workspace_size(batch: int, num_q_heads: int, max_pages_per_seq: int, page_size: int,
                                  window: int, num_splits: int = 0) -> int:
    return int(load().cai_mqa_decode_workspace_size(batch, num_q_heads, max_pages_per_seq, page_size, window,
                                                     num_splits))


def _pool_array(pools: Sequence[KVPool]):
    arr = (cai_kv_pool * len(pools))()
    for i, p in enumerate(pools):
        arr[i] = p.struct
    return arr


def cai_mqa_decode(pools: Sequence[KVPool], layer_to_pool: Sequence[int], layer: int, q: torch.Tensor,
                   block_table: torch.Tensor, ctx_len: torch.Tensor, window: int, softmax_scale: float,
                   num_splits: int, workspace: Optional[torch.Tensor], out: torch.Tensor,
                   lse_out: Optional[torch.Tensor] = None, err_flag: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """One decode step of one layer: q bf16 [batch][Hq][128] -> out fp32 [batch][Hq][128]."""
    batch, hq = q.shape[0], q.shape[1]
    l2p = (ctypes.c_int32 * len(layer_to_pool))(*layer_to_pool)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().cai_mqa_decode(
        _pool_array(pools), len(pools), l2p, len(layer_to_pool), layer,
        _ptr(q, "q", (torch.bfloat16, torch.int16), (batch, hq, HEAD_DIM)), batch, hq,
        _ptr(block_table, "block_table", torch.int32), block_table.shape[-1],
        _ptr(ctx_len, "ctx_len", torch.int32, (batch,)), window, float(softmax_scale), num_splits,
        _ptr(workspace, "workspace"), ws_bytes, _ptr(out, "out", torch.float32, (batch, hq, HEAD_DIM)),
        _ptr(lse_out, "lse_out", torch.float32, (batch, hq)), _ptr(err_flag, "err_flag", torch.int32),
        _stream(stream))
    _check(st, "cai_mqa_decode")


def cai_mqa_decode_layers_workspace_size(batch: int, num_q_heads: int, max_pages_per_seq: int, page_size: int,
                                         windows: Sequence[int], num_splits: int = 0) -> int:
    w = (ctypes.c_int32 * len(windows))(*windows)
    return int(load().cai_mqa_decode_layers_workspace_size(batch, num_q_heads, max_pages_per_seq, page_size,
                                                            len(windows), w, num_splits))


def cai_mqa_decode_layers(pools: Sequence[KVPool], layer_to_pool: Sequence[int], windows: Sequence[int],
                          qs: Sequence[torch.Tensor], block_tables: Sequence[torch.Tensor], ctx_len: torch.Tensor,
                          softmax_scale: float, num_splits: int, workspace: Optional[torch.Tensor],
                          outs: Sequence[torch.Tensor], lse_outs: Optional[Sequence[Optional[torch.Tensor]]] = None,
                          err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """One decode step of several layers in one launch: qs[l] bf16 [batch][Hq][128] -> outs[l] fp32."""
    n = len(layer_to_pool)
    if not (len(windows) == len(qs) == len(block_tables) == len(outs) == n):
        raise ValueError("layer_to_pool, windows, qs, block_tables and outs must have one entry per layer")
    if lse_outs is not None and len(lse_outs) != n:
        raise ValueError("lse_outs must have one entry per layer")
    batch, hq = qs[0].shape[0], qs[0].shape[1]
    max_pages = block_tables[0].shape[-1]
    for t in block_tables:
        if t.shape[-1] != max_pages:
            raise ValueError("block tables of one call must have the same width")
    l2p = (ctypes.c_int32 * n)(*layer_to_pool)
    win = (ctypes.c_int32 * n)(*windows)
    q_ptrs = (ctypes.c_void_p * n)(*[_ptr(q, "q", (torch.bfloat16, torch.int16), (batch, hq, HEAD_DIM)) for q in qs])
    t_ptrs = (ctypes.c_void_p * n)(*[_ptr(t, "block_table", torch.int32) for t in block_tables])
    o_ptrs = (ctypes.c_void_p * n)(*[_ptr(o, "out", torch.float32, (batch, hq, HEAD_DIM)) for o in outs])
    l_ptrs = None
    if lse_outs is not None:
        l_ptrs = (ctypes.c_void_p * n)(*[_ptr(t, "lse_out", torch.float32, (batch, hq)) for t in lse_outs])
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().cai_mqa_decode_layers(
        _pool_array(pools), len(pools), l2p, n, win, q_ptrs, batch, hq, t_ptrs, max_pages,
        _ptr(ctx_len, "ctx_len", torch.int32, (batch,)), float(softmax_scale), num_splits,
        _ptr(workspace, "workspace"), ws_bytes, o_ptrs, l_ptrs, _ptr(err_flag, "err_flag", torch.int32),
        _stream(stream))
    _check(st, "cai_mqa_decode_layers")


def cai_mqa_decode_no_alloc(pools: Sequence[KVPool], layer_to_pool: Sequence[int], layer: int, q: torch.Tensor,
                            block_table: torch.Tensor, ctx_len: torch.Tensor, window: int, softmax_scale: float,
                            num_splits: int, out: torch.Tensor, lse_out: Optional[torch.Tensor] = None,
                            err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """cai_mqa_decode for callers that cannot allocate: split partials live in the library's own scratch."""
    batch, hq = q.shape[0], q.shape[1]
    l2p = (ctypes.c_int32 * len(layer_to_pool))(*layer_to_pool)
    st = load().cai_mqa_decode_no_alloc(
        _pool_array(pools), len(pools), l2p, len(layer_to_pool), layer,
        _ptr(q, "q", (torch.bfloat16, torch.int16), (batch, hq, HEAD_DIM)), batch, hq,
        _ptr(block_table, "block_table", torch.int32), block_table.shape[-1],
        _ptr(ctx_len, "ctx_len", torch.int32, (batch,)), window, float(softmax_scale), num_splits,
        _ptr(out, "out", torch.float32, (batch, hq, HEAD_DIM)), _ptr(lse_out, "lse_out", torch.float32, (batch, hq)),
        _ptr(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "cai_mqa_decode_no_alloc")


def cai_mqa_prefill_workspace_size(batch: int, max_pages_per_seq: int, page_size: int) -> int:
    return int(load().cai_mqa_prefill_workspace_size(batch, max_pages_per_seq, page_size))


def cai_mqa_prefill_chunk(pool: KVPool, q: torch.Tensor, block_table: torch.Tensor, prefix_len: torch.Tensor,
                          window: int, softmax_scale: float, workspace: torch.Tensor, out: torch.Tensor,
                          lse_out: Optional[torch.Tensor] = None, err_flag: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """Attention of n_new appended tokens on a reused prefix: q bf16 [batch][n_new][Hq][128]."""
    batch, n_new, hq = q.shape[0], q.shape[1], q.shape[2]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().cai_mqa_prefill_chunk(
        ctypes.byref(pool.struct), _ptr(q, "q", (torch.bfloat16, torch.int16), (batch, n_new, hq, HEAD_DIM)), batch,
        n_new, hq, _ptr(block_table, "block_table", torch.int32), block_table.shape[-1],
        _ptr(prefix_len, "prefix_len", torch.int32, (batch,)), window, float(softmax_scale),
        _ptr(workspace, "workspace"), ws_bytes, _ptr(out, "out", torch.float32, (batch, n_new, hq, HEAD_DIM)),
        _ptr(lse_out, "lse_out", torch.float32, (batch, n_new, hq)), _ptr(err_flag, "err_flag", torch.int32),
        _stream(stream))
    _check(st, "cai_mqa_prefill_chunk")


def cai_gqa_decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, max_pages_per_seq: int,
                                  page_size: int, window: int, num_splits: int = 0) -> int:
    return int(load().cai_gqa_decode_workspace_size(batch, num_q_heads, num_kv_heads, max_pages_per_seq, page_size,
                                                    window, num_splits))


def cai_gqa_decode(kv_pools: Sequence[KVPool], q: torch.Tensor, block_table: torch.Tensor, ctx_len: torch.Tensor,
                   window: int, softmax_scale: float, num_splits: int, workspace: torch.Tensor, out: torch.Tensor,
                   lse_out: Optional[torch.Tensor] = None, err_flag: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """Grouped-query decode: query heads [j*G, (j+1)*G) read kv_pools[j], G = Hq / len(kv_pools)."""
    batch, hq = q.shape[0], q.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().cai_gqa_decode(
        _pool_structs(kv_pools), len(kv_pools), _ptr(q, "q", (torch.bfloat16, torch.int16), (batch, hq, HEAD_DIM)),
        batch, hq, _ptr(block_table, "block_table", torch.int32), block_table.shape[-1],
        _ptr(ctx_len, "ctx_len", torch.int32, (batch,)), window, float(softmax_scale), num_splits,
        _ptr(workspace, "workspace"), ws_bytes, _ptr(out, "out", torch.float32, (batch, hq, HEAD_DIM)),
        _ptr(lse_out, "lse_out", torch.float32, (batch, hq)), _ptr(err_flag, "err_flag", torch.int32),
        _stream(stream))
    _check(st, "cai_gqa_decode")


def cai_mqa_prefill_varlen(pool: KVPool, q: torch.Tensor, q_offsets: torch.Tensor, max_new: int,
                           block_table: torch.Tensor, prefix_len: torch.Tensor, window: int, softmax_scale: float,
                           workspace: torch.Tensor, out: torch.Tensor, lse_out: Optional[torch.Tensor] = None,
                           err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """Mixed batch in one launch: sequence b's new tokens are rows q_offsets[b] .. q_offsets[b+1]
    of the packed q bf16 [total_new][Hq][128] (decode steps are one-row sequences)."""
    total, hq = q.shape[0], q.shape[1]
    batch = q_offsets.shape[0] - 1
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().cai_mqa_prefill_varlen(
        ctypes.byref(pool.struct), _ptr(q, "q", (torch.bfloat16, torch.int16), (total, hq, HEAD_DIM)), batch,
        _ptr(q_offsets, "q_offsets", torch.int32, (batch + 1,)), total, int(max_new), hq,
        _ptr(block_table, "block_table", torch.int32), block_table.shape[-1],
        _ptr(prefix_len, "prefix_len", torch.int32, (batch,)), window, float(softmax_scale),
        _ptr(workspace, "workspace"), ws_bytes, _ptr(out, "out", torch.float32, (total, hq, HEAD_DIM)),
        _ptr(lse_out, "lse_out", torch.float32, (total, hq)), _ptr(err_flag, "err_flag", torch.int32),
        _stream(stream))
    _check(st, "cai_mqa_prefill_varlen")


# ----------------------------------------------------------------------------- cross-turn host KV cache

def _i32_host(a) -> "ctypes.Array":
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def cai_set_wait_limit_ns(ns: int) -> None:
    """Limit of the kernels' bounded waits in nanoseconds (0: the default, 2 s); for failure tests."""
    load().cai_set_wait_limit_ns(int(ns))


def cai_set_fault_injection(stage: int) -> None:
    """Every CTA skips the load of its `stage`-th K/V stage (decode) or K tile (prefill); -1: off."""
    load().cai_set_fault_injection(int(stage))


def cai_host_cache_create(page_size: int, num_buffers: int, capacity_pages: int, head_dim: int = HEAD_DIM) -> int:
    h = load().cai_host_cache_create(page_size, head_dim, num_buffers, capacity_pages)
    if not h:
        raise CaiError(CAI_ERR_INVALID_ARG, "cai_host_cache_create")
    return h


def cai_host_cache_destroy(cache: int) -> None:
    load().cai_host_cache_destroy(cache)


def cai_host_cache_match(cache: int, tokens) -> int:
    keep, ptr = _i32_host(tokens)
    return int(load().cai_host_cache_match(cache, ptr, len(keep)))


def _pool_structs(pools):
    arr = (cai_kv_pool * len(pools))()
    for i, p in enumerate(pools):
        arr[i] = p.struct if isinstance(p, KVPool) else p
    return arr


def cai_host_cache_restore(cache: int, tokens, n_tokens: int, pools, block_table_row, stream=None) -> None:
    keep, ptr = _i32_host(tokens)
    tkeep, tptr = _i32_host(block_table_row)
    st = load().cai_host_cache_restore(cache, ptr, n_tokens, _pool_structs(pools), tptr,
                                       _stream(stream) if torch.cuda.is_available() else None)
    _check(st, "cai_host_cache_restore")


def cai_host_cache_restore_batch(cache: int, tokens, n_tokens, pools, block_table_rows, stream=None) -> None:
    """cai_host_cache_restore for several sequences in one call (tokens[i], n_tokens[i], block_table_rows[i])."""
    keeps = [_i32_host(t) for t in tokens]
    tkeeps = [_i32_host(r) for r in block_table_rows]
    n = len(keeps)
    tok_ptrs = (ctypes.c_void_p * max(n, 1))(*[p for _, p in keeps])
    row_ptrs = (ctypes.c_void_p * max(n, 1))(*[p for _, p in tkeeps])
    counts = np.ascontiguousarray(np.asarray(n_tokens, dtype=np.int32))
    st = load().cai_host_cache_restore_batch(cache, n, tok_ptrs, counts.ctypes.data_as(ctypes.c_void_p),
                                             _pool_structs(pools), row_ptrs,
                                             _stream(stream) if torch.cuda.is_available() else None)
    _check(st, "cai_host_cache_restore_batch")


def cai_host_cache_store(cache: int, tokens, pools, block_table_row, stream=None) -> None:
    keep, ptr = _i32_host(tokens)
    tkeep, tptr = _i32_host(block_table_row)
    st = load().cai_host_cache_store(cache, ptr, len(keep), _pool_structs(pools), tptr,
                                     _stream(stream) if torch.cuda.is_available() else None)
    _check(st, "cai_host_cache_store")


def cai_host_cache_stats(cache: int) -> dict:
    v = [ctypes.c_int64() for _ in range(4)]
    load().cai_host_cache_stats(cache, *[ctypes.byref(x) for x in v])
    return dict(zip(("hits", "misses", "pages_cached", "evictions"), (x.value for x in v)))


def cai_ring_pages(window: int, page_size: int, max_new_tokens: int = 1) -> int:
    """Pages per sequence of a local buffer's ring (0 for invalid arguments)."""
    return int(load().cai_ring_pages(window, page_size, max_new_tokens))


def cai_ring_table_row(ring_ids, hi: int, page_size: int, max_pages_per_seq: int) -> np.ndarray:
    """One block-table row (host int32 [max_pages_per_seq]) mapping the live pages of a
    sequence written up to `hi` into its ring; freed and unwritten entries are -1."""
    ids = np.ascontiguousarray(np.asarray(ring_ids, dtype=np.int32))
    row = np.empty(max_pages_per_seq, dtype=np.int32)
    st = load().cai_ring_table_row(row.ctypes.data, max_pages_per_seq, ids.ctypes.data, len(ids), hi, page_size)
    _check(st, "cai_ring_table_row")
    return row

"""Harness shared by the GPU tests and bench.py: synthetic paged KV caches and
step inputs for the pages' workloads, built on the GPU through the public
binding (the fill uses cai_kv_append itself, over seeded fp32 K/V).

The oracle side regenerates the same inputs on the host from the same seeds
(synth.kv_rows / synth.q_rows); nothing computed here feeds the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import int8_mqa_decode_gb300 as cai
import synth
import synth.gpu as sgpu

TABLE_STREAM = 77


class PagedCache:
    """KV buffers (one pool each), one shared block table and per-sequence lengths."""

    def __init__(self, w: synth.Workload, device: str = "cuda", shuffle: bool = True, sentinel: int | None = None,
                 spare_pages: int = 0, max_pages_per_seq: int | None = None):
        self.w = w
        self.device = device
        mp = max_pages_per_seq or w.max_pages_per_seq
        self.table_np, self.num_pages = synth.block_table(w.seed, TABLE_STREAM, w.ctx_len, w.page_size, mp,
                                                          shuffle=shuffle, spare_pages=spare_pages)
        self.table = torch.from_numpy(self.table_np).to(device)
        self.pools = [cai.KVPool(self.num_pages, w.page_size, device=device) for _ in range(w.num_buffers)]
        if sentinel is not None:
            for p in self.pools:
                p.pages.fill_(sentinel)
        self.ctx_len_np = np.asarray(w.ctx_len, dtype=np.int64)
        self.ctx_len = torch.from_numpy(self.ctx_len_np.astype(np.int32)).to(device)

    @property
    def max_pages_per_seq(self) -> int:
        return self.table.shape[1]

    def fill(self, upto=None, max_chunk: int = 1 << 16) -> None:
        """Append positions [0, upto[b]) of every sequence in every buffer (default: all but the step's tokens)."""
        w = self.w
        upto = (self.ctx_len_np - w.n_new) if upto is None else np.asarray(upto)
        start = torch.zeros(1, dtype=torch.int32, device=self.device)
        for buf, pool in enumerate(self.pools):
            for b in range(w.batch):
                n_total = int(upto[b])
                for p0 in range(0, n_total, max_chunk):
                    n = min(max_chunk, n_total - p0)
                    k = torch.empty(1, n, 128, dtype=torch.float32, device=self.device)
                    v = torch.empty_like(k)
                    sgpu.normal_rows(k, w.seed, synth.stream_k(buf), b, p_const=p0)
                    sgpu.normal_rows(v, w.seed, synth.stream_v(buf), b, p_const=p0)
                    start.fill_(p0)
                    cai.cai_kv_append(pool, k, v, self.table[b:b + 1], start)

    def step_kv(self, buf: int, n_new: int | None = None):
        """fp32 K, V [B][n_new][128] of the step's new tokens (positions ctx_len - n_new ..) and their start."""
        w = self.w
        n_new = w.n_new if n_new is None else n_new
        start = (self.ctx_len - n_new).to(torch.int32)
        k = torch.empty(w.batch, n_new, 128, dtype=torch.float32, device=self.device)
        v = torch.empty_like(k)
        sgpu.normal_rows(k, w.seed, synth.stream_k(buf), 0, pos=start)
        sgpu.normal_rows(v, w.seed, synth.stream_v(buf), 0, pos=start)
        return k, v, start

    def decode_q(self, layer: int) -> torch.Tensor:
        w = self.w
        q = torch.empty(w.batch, w.num_q_heads, 128, dtype=torch.bfloat16, device=self.device)
        return sgpu.q_rows(q, w.seed, synth.stream_q(layer), 0)

    def prefill_q(self) -> torch.Tensor:
        w = self.w
        q = torch.empty(w.batch, w.n_new * w.num_q_heads, 128, dtype=torch.bfloat16, device=self.device)
        sgpu.q_rows(q, w.seed, synth.STREAM_Q_PREFILL, 0)
        return q.view(w.batch, w.n_new, w.num_q_heads, 128)

    def append_step(self, err=None) -> None:
        """Append the step's new tokens to every buffer."""
        for buf, pool in enumerate(self.pools):
            k, v, start = self.step_kv(buf)
            cai.cai_kv_append(pool, k, v, self.table, start, err_flag=err)

    def workspace(self, layer: int, num_splits: int = 0) -> torch.Tensor | None:
        w = self.w
        n = cai.cai_mqa_decode_workspace_size(w.batch, w.num_q_heads, self.max_pages_per_seq, w.page_size,
                                              w.layer_windows[layer], num_splits)
        return torch.zeros(n, dtype=torch.uint8, device=self.device)  # the header must start at zero

    def prefill_workspace(self) -> torch.Tensor:
        n = cai.cai_mqa_prefill_workspace_size(self.w.batch, self.max_pages_per_seq, self.w.page_size)
        return torch.empty(n, dtype=torch.uint8, device=self.device)

    def prefill(self, q: torch.Tensor, out: torch.Tensor, lse: torch.Tensor | None = None, workspace=None,
                window: int | None = None, err=None) -> None:
        """Attention of the step's n_new tokens (already appended) on the prefix ctx_len - n_new."""
        w = self.w
        if workspace is None:
            workspace = self.prefill_workspace()
        prefix = (self.ctx_len - w.n_new).to(torch.int32)
        cai.cai_mqa_prefill_chunk(self.pools[0], q, self.table, prefix, w.layer_windows[0] if window is None else window,
                                  w.softmax_scale, workspace, out, lse, err)

    def decode(self, layer: int, q: torch.Tensor, out: torch.Tensor, lse: torch.Tensor | None = None,
               num_splits: int = 0, workspace=None, err=None) -> None:
        w = self.w
        if workspace is None:
            workspace = self.workspace(layer, num_splits)
        cai.cai_mqa_decode(self.pools, w.layer_to_buffer, layer, q, self.table, self.ctx_len,
                           w.layer_windows[layer], w.softmax_scale, num_splits, workspace, out, lse, err)

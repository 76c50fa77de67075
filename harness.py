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
    """KV buffers (one pool each), their block tables and per-sequence lengths.

    By default every buffer has a full pool and all share one block table.  With
    `local_ring`, a buffer read only by local layers keeps each sequence in a ring of
    cai_ring_pages(window, P, n) pages (n = the most tokens one call writes): its pool
    holds batch * ring pages and its table maps only the live pages (-1 elsewhere), so
    any kernel read of a freed page raises CAI_DEVERR_PAGE.
    """

    def __init__(self, w: synth.Workload, device: str = "cuda", shuffle: bool = True, sentinel: int | None = None,
                 spare_pages: int = 0, max_pages_per_seq: int | None = None, local_ring: bool = False,
                 ring_new_tokens: int = 1):
        self.w = w
        self.device = device
        mp = max_pages_per_seq or w.max_pages_per_seq
        self.table_np, self.num_pages = synth.block_table(w.seed, TABLE_STREAM, w.ctx_len, w.page_size, mp,
                                                          shuffle=shuffle, spare_pages=spare_pages)
        self.table = torch.from_numpy(self.table_np).to(device)
        self.ctx_len_np = np.asarray(w.ctx_len, dtype=np.int64)
        self.ctx_len = torch.from_numpy(self.ctx_len_np.astype(np.int32)).to(device)
        self.ring = [0] * w.num_buffers          # ring pages per sequence (0 = full pool)
        self.ring_ids = [None] * w.num_buffers   # host [batch][ring] page ids
        pool_pages = [self.num_pages] * w.num_buffers
        if local_ring:
            n_new = max(int(ring_new_tokens), int(w.n_new))
            for buf in range(w.num_buffers):
                wins = [w.layer_windows[l] for l in range(len(w.layer_windows)) if w.layer_to_buffer[l] == buf]
                if wins and min(wins) > 0:
                    r = cai.cai_ring_pages(max(wins), w.page_size, n_new)
                    self.ring[buf] = r
                    perm = synth.permutation(w.seed, TABLE_STREAM + 1 + buf, w.batch * r) if shuffle \
                        else np.arange(w.batch * r)
                    self.ring_ids[buf] = np.asarray(perm, dtype=np.int32).reshape(w.batch, r)
                    pool_pages[buf] = w.batch * r
        self.pools = [cai.KVPool(pool_pages[buf], w.page_size, device=device) for buf in range(w.num_buffers)]
        if sentinel is not None:
            for p in self.pools:
                p.pages.fill_(sentinel)
        # ring tables used while filling (every logical page mapped to its slot) and per step (live pages only)
        self.ring_fill_tables = {b: self._ring_table(b, None) for b in range(w.num_buffers) if self.ring[b]}
        self.ring_tables = {b: self._ring_table(b, self.ctx_len_np) for b in range(w.num_buffers) if self.ring[b]}

    @property
    def tables(self) -> list:
        """Block table of each buffer for the step's calls (the shared `table` for full pools)."""
        return [self.ring_tables.get(b, self.table) for b in range(self.w.num_buffers)]

    def _ring_table(self, buf: int, hi) -> torch.Tensor:
        """Ring table of a buffer: live pages for lengths `hi` (None: every logical page mapped)."""
        w, r, mp = self.w, self.ring[buf], self.table.shape[1]
        rows = np.empty((w.batch, mp), dtype=np.int32)
        for b in range(w.batch):
            if hi is None:
                rows[b] = self.ring_ids[buf][b][np.arange(mp) % r]
            else:
                rows[b] = cai.cai_ring_table_row(self.ring_ids[buf][b], int(hi[b]), w.page_size, mp)
        return torch.from_numpy(rows).to(self.device)

    def pool_bytes(self) -> int:
        return sum(p.num_pages for p in self.pools) * cai.cai_page_bytes(self.w.page_size)

    @property
    def max_pages_per_seq(self) -> int:
        return self.table.shape[1]

    def fill(self, upto=None, max_chunk: int = 1 << 16) -> None:
        """Append positions [0, upto[b]) of every sequence in every buffer (default: all but the step's tokens).
        A ring buffer is filled in chunks of at most (ring - 1) pages, so no chunk writes one slot twice."""
        w = self.w
        upto = (self.ctx_len_np - w.n_new) if upto is None else np.asarray(upto)
        start = torch.zeros(1, dtype=torch.int32, device=self.device)
        for buf, pool in enumerate(self.pools):
            chunk = max_chunk if not self.ring[buf] else min(max_chunk, (self.ring[buf] - 1) * w.page_size)
            table = self.ring_fill_tables.get(buf, self.table)
            for b in range(w.batch):
                n_total = int(upto[b])
                for p0 in range(0, n_total, chunk):
                    n = min(chunk, n_total - p0)
                    k = torch.empty(1, n, 128, dtype=torch.float32, device=self.device)
                    v = torch.empty_like(k)
                    sgpu.normal_rows(k, w.seed, synth.stream_k(buf), b, p_const=p0)
                    sgpu.normal_rows(v, w.seed, synth.stream_v(buf), b, p_const=p0)
                    start.fill_(p0)
                    cai.cai_kv_append(pool, k, v, table[b:b + 1], start)

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
        """Append the step's new tokens to every buffer (one launch)."""
        kv = [self.step_kv(buf) for buf in range(len(self.pools))]
        cai.cai_kv_append_pools(self.pools, [k for k, _, _ in kv], [v for _, v, _ in kv], self.tables,
                                [s for _, _, s in kv], err_flag=err)

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
        cai.cai_mqa_prefill_chunk(self.pools[0], q, self.tables[0], prefix,
                                  w.layer_windows[0] if window is None else window, w.softmax_scale, workspace, out,
                                  lse, err)

    def layers_workspace(self, num_splits: int = 0) -> torch.Tensor:
        w = self.w
        n = cai.cai_mqa_decode_layers_workspace_size(w.batch, w.num_q_heads, self.max_pages_per_seq, w.page_size,
                                                     list(w.layer_windows), num_splits)
        return torch.zeros(n, dtype=torch.uint8, device=self.device)  # the header must start at zero

    def decode_layers(self, qs, outs, lses=None, num_splits: int = 0, workspace=None, err=None) -> None:
        """Every layer of the step in one launch (qs[l], outs[l] as for decode)."""
        w = self.w
        if workspace is None:
            workspace = self.layers_workspace(num_splits)
        tables = [self.tables[w.layer_to_buffer[layer]] for layer in range(len(w.layer_windows))]
        cai.cai_mqa_decode_layers(self.pools, w.layer_to_buffer, list(w.layer_windows), qs, tables, self.ctx_len,
                                  w.softmax_scale, num_splits, workspace, outs, lses, err)

    def decode(self, layer: int, q: torch.Tensor, out: torch.Tensor, lse: torch.Tensor | None = None,
               num_splits: int = 0, workspace=None, err=None) -> None:
        w = self.w
        if workspace is None:
            workspace = self.workspace(layer, num_splits)
        cai.cai_mqa_decode(self.pools, w.layer_to_buffer, layer, q, self.tables[w.layer_to_buffer[layer]],
                           self.ctx_len, w.layer_windows[layer], w.softmax_scale, num_splits, workspace, out, lse, err)

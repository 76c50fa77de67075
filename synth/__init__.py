"""Seeded synthetic inputs shared by the oracle side and the GPU side.

This module holds input generation only: no quantization, no attention, no
page layout.  Both sides draw the same numbers from the same counters:

* ``splitmix64``: the counter-based generator of Steele, Lea and Flood
  ("Fast splittable pseudorandom number generators", OOPSLA 2014), written
  here from its published definition: the n-th output for seed ``s`` is the
  64-bit finaliser applied to ``s + (n + 1) * 0x9E3779B97F4A7C15``.
* ``normal``: an Irwin-Hall(12) approximation of N(0, 1).  Each value sums
  twelve 20-bit uniforms (three from each of four splitmix64 outputs),
  subtracts 6 * 2**20 and divides by 2**20.  Every step is exact in fp32, so
  the CPU and the GPU produce identical bits.  Variance is 1 and the tails are
  cut at +-6.
* queries are those normals rounded to bf16 (round to nearest, ties to even).

A value is addressed by ``(stream, b, p, d)``: a tensor id, a sequence, a
position (or token*heads + head for queries) and a channel.  The counter is
``((stream << 40) | (b << 27) | (p << 7) | d) * 4 + r`` for r in 0..3.

The GPU twin of these generators is ``synth_gpu.cu`` in this folder; a test
checks that both give the same bits.

Workload recipes (lengths, block tables) for the pages' five workloads are at
the bottom of this file.  Lengths and block tables are made on the host, once,
and uploaded; the same arrays feed the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK20 = np.uint64(0xFFFFF)

# Tensor ids ("streams") used by the workloads.
def stream_k(buffer: int) -> int:
    return 2 * buffer


def stream_v(buffer: int) -> int:
    return 2 * buffer + 1


def stream_q(layer: int) -> int:
    return 1000 + layer


STREAM_Q_PREFILL = 2000
MAX_B = 1 << 13
MAX_P = 1 << 20
MAX_D = 1 << 7


def splitmix64(seed: int, n: np.ndarray) -> np.ndarray:
    """n-th splitmix64 output for ``seed`` (n: uint64 array)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (n.astype(np.uint64) + np.uint64(1)) * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _index(stream: int, b, p, d) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint64)
    p = np.asarray(p, dtype=np.uint64)
    d = np.asarray(d, dtype=np.uint64)
    return (np.uint64(stream) << np.uint64(40)) | (b << np.uint64(27)) | (p << np.uint64(7)) | d


def normal_at(seed: int, stream: int, b, p, d) -> np.ndarray:
    """Irwin-Hall(12) normals at broadcast coordinates (b, p, d) -> float32."""
    idx = _index(stream, b, p, d)
    acc = np.zeros(idx.shape, dtype=np.int64)
    for r in range(4):
        h = splitmix64(seed, idx * np.uint64(4) + np.uint64(r))
        acc += (h & _MASK20).astype(np.int64)
        acc += ((h >> np.uint64(20)) & _MASK20).astype(np.int64)
        acc += ((h >> np.uint64(40)) & _MASK20).astype(np.int64)
    acc -= 6 << 20
    return acc.astype(np.float32) / np.float32(1 << 20)


def kv_rows(seed: int, stream: int, b: int, p0: int, n: int, dim: int = 128) -> np.ndarray:
    """fp32 rows [n][dim] of sequence b at positions p0 .. p0+n-1."""
    assert 0 <= b < MAX_B and 0 <= p0 and p0 + n <= MAX_P and dim <= MAX_D
    p = np.arange(p0, p0 + n, dtype=np.uint64)[:, None]
    d = np.arange(dim, dtype=np.uint64)[None, :]
    return normal_at(seed, stream, b, p, d)


def bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32)


def q_rows(seed: int, stream: int, b: int, rows: int, dim: int = 128) -> np.ndarray:
    """bf16 bits [rows][dim] of sequence b; row r is coordinate p = r.

    Decode queries use rows = heads; prefill queries use row = token*heads + head.
    """
    assert 0 <= b < MAX_B and rows <= MAX_P and dim <= MAX_D
    p = np.arange(rows, dtype=np.uint64)[:, None]
    d = np.arange(dim, dtype=np.uint64)[None, :]
    return bf16_bits_rne(normal_at(seed, stream, b, p, d))


# ---------------------------------------------------------------------------
# Host-side recipes: lengths and block tables.
# ---------------------------------------------------------------------------

def uniform01(seed: int, stream: int, n: int) -> np.ndarray:
    """n doubles in [0, 1) from splitmix64 (53-bit mantissas)."""
    h = splitmix64(seed, (np.uint64(stream) << np.uint64(40)) + np.arange(n, dtype=np.uint64))
    return (h >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive)."""
    u = uniform01(seed, stream, n)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64).clip(lo, hi)


def lognormal_int(seed: int, stream: int, n: int, median: float, sigma: float, lo: int, hi: int) -> np.ndarray:
    """n integers, lognormal(ln median, sigma) by Box-Muller, rounded and clipped to [lo, hi]."""
    u1 = uniform01(seed, stream, n)
    u2 = uniform01(seed, stream + 1, n)
    z = np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)
    return np.clip(np.rint(median * np.exp(sigma * z)), lo, hi).astype(np.int64)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Seeded Fisher-Yates permutation of 0..n-1."""
    u = uniform01(seed, stream, n)
    perm = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(u[i] * (i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


def block_table(seed: int, stream: int, capacity_tokens: np.ndarray, page_size: int,
                max_pages_per_seq: int, shuffle: bool = True, spare_pages: int = 0):
    """Assign physical pages to sequences.

    Each sequence b gets ceil(capacity_tokens[b] / page_size) pages, taken in
    order from a (seeded, optionally shuffled) list of all pages.  Unused table
    entries are -1.  Returns (table int32 [B][max_pages_per_seq], num_pages).
    """
    need = [(int(c) + page_size - 1) // page_size for c in capacity_tokens]
    assert max(need) <= max_pages_per_seq
    total = sum(need) + spare_pages
    order = permutation(seed, stream, total) if shuffle else np.arange(total)
    table = np.full((len(need), max_pages_per_seq), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = order[k:k + n]
        k += n
    return table, total


@dataclass
class Workload:
    """One of the pages' five workloads, with seeded lengths and pages."""
    name: str
    batch: int
    num_q_heads: int
    page_size: int
    ctx_len: np.ndarray               # [B] tokens cached after this step's append (includes the current token)
    layer_windows: list               # window per layer (0 = global)
    layer_to_buffer: list             # buffer per layer
    n_new: int = 1                    # tokens appended per sequence per buffer in the step
    seed: int = 1000
    head_dim: int = 128
    softmax_scale: float = 1.0 / math.sqrt(128.0)
    num_splits: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def num_buffers(self) -> int:
        return max(self.layer_to_buffer) + 1

    @property
    def max_pages_per_seq(self) -> int:
        return int((int(self.ctx_len.max()) + self.page_size - 1) // self.page_size)


def workload(config: int, seed: int | None = None, sigma: float = 1.0, batch: int | None = None) -> Workload:
    """The five workloads (1-based, in the order the pages' workload list gives them).

    ``batch`` overrides the batch size (used to shrink a workload for a test).
    """
    s = (1000 + config) if seed is None else seed
    if config == 1:
        B = batch or 4
        L = uniform_int(s, 1, B, 64, 512)
        return Workload("tiny-global B=4 Hq=8 L~U[64,512] P=16", B, 8, 16, L, [0], [0], seed=s)
    if config == 2:
        B = batch or 64
        L = uniform_int(s, 1, B, 1024, 8192)
        return Workload("local-decode B=64 Hq=32 L~U[1024,8192] W=1024 P=16", B, 32, 16, L, [1024], [0], seed=s)
    if config == 3:
        B = batch or 256
        L = lognormal_int(s, 1, B, 4096.0, sigma, 256, 32768)
        return Workload("hybrid-6-layer B=256 Hq=32 L~lognormal(ln4096,%g)[256,32768] W=1024x5+global P=16" % sigma,
                        B, 32, 16, L, [1024] * 5 + [0], [0, 0, 1, 1, 2, 3], seed=s)
    if config == 4:
        B = batch or 16
        L = np.full(B, 8192 + 256, dtype=np.int64)
        return Workload("append-prefill B=16 prefix=8192 n_new=256 Hq=32 P=16", B, 32, 16, L, [0], [0],
                        n_new=256, seed=s, extra={"prefix": 8192})
    if config == 5:
        B = batch or 1024
        L = uniform_int(s, 1, B, 16384, 131072)
        return Workload("long-global B=1024 Hq=64 L~U[16384,131072] P=64", B, 64, 64, L, [0], [0], seed=s)
    raise ValueError(f"unknown workload {config}")

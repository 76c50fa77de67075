"""Oracle for the int8 MQA paged decode path: plain, slow, CPU only.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
library never imports, links or calls it, and it never calls the CUDA library.
Inputs come from ``synth`` (seeded generators only); every number here is
computed from those inputs by the arithmetic below and in ``oracle.c``.

What is computed, and from which passage of the pages:

* ``quantize_rows``: int8 KV cache ("Character.AI: inference optimization",
  05 Quantization and cost).  Reading: symmetric per-token absmax, fp32 scale
  s = absmax/127, code = round-half-even(x/s) clamped to [-127, 127], both
  divisions single IEEE fp32 operations; a zero scale (absmax 0, or absmax/127
  underflowing to 0) gives zero codes.
* ``attend``: softmax attention of one query per head over cached keys and
  values ("Como funciona a inferencia de IA", "Por que o cache KV existe"),
  with one shared K/V head (Multi-Query Attention, technique table of section
  03), in float64.
* ``merge_splits``: softmax attention over a union of disjoint parts of the
  attended set, from each part's normalised output and log-sum-exp (the
  algebra a split-KV decode relies on; the definition itself never splits).
* ``attended_range``: global layers see every cached token; local layers see
  the last ``window`` positions, the current token included (hybrid attention
  with horizon 1024, technique table of section 03).
* ``pool_write`` / ``pool_read``: the paged layout (PagedAttention, section
  "1. PagedAttention" of the Red Hat page): fixed-size blocks anywhere in a
  pool plus a per-sequence table of block ids.  Byte layout of one page of P
  tokens and head_dim d (the pages fix none; this is the library's): K codes
  int8 [P][d] (token-major), V codes int8 [d][P] (channel-major: the P codes
  of channel c are contiguous), K scales fp32 [P], V scales fp32 [P]; token at
  position p of a sequence sits in page table[p // P], slot p % P.
* ``prefill_ranges``: new tokens appended on top of a reused prefix (prefix
  caching, section "3. Cache de prefixo"; cross-turn cache, section 04): new
  token i at absolute position p0+i attends keys 0..p0+i, all of them read
  back from the int8 cache.
* ``kv_cache_bytes_per_token``: the KV-size formula of the section "Qual e o
  tamanho real do cache KV?".

Every function here is pinned by tests in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            lib.oracle_quantize_rows.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P]
            lib.oracle_quantize_rows.restype = None
            lib.oracle_dequantize.argtypes = [P, P, ctypes.c_int64, ctypes.c_int32, P]
            lib.oracle_dequantize.restype = None
            lib.oracle_attend.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_int64, ctypes.c_double,
                                          P, P]
            lib.oracle_attend.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# Quantizer and attention (compiled C, see oracle.c)
# ---------------------------------------------------------------------------

def quantize_rows(x: np.ndarray):
    """x float32 [n][d] -> (codes int8 [n][d], scales float32 [n])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n, d = x.shape
    codes = np.empty((n, d), dtype=np.int8)
    scales = np.empty(n, dtype=np.float32)
    _load().oracle_quantize_rows(_ptr(x), n, d, _ptr(codes), _ptr(scales))
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes int8 [T][d], scales float32 [T] -> float64 [T][d] (exact)."""
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    T, d = codes.shape
    out = np.empty((T, d), dtype=np.float64)
    _load().oracle_dequantize(_ptr(codes), _ptr(scales), T, d, _ptr(out))
    return out


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, c: float):
    """q float64 [Hq][d]; k, v float64 [T][d] -> (out float64 [Hq][d], lse float64 [Hq])."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    Hq, d = q.shape
    T = k.shape[0]
    assert k.shape == (T, d) and v.shape == (T, d)
    out = np.empty((Hq, d), dtype=np.float64)
    lse = np.empty(Hq, dtype=np.float64)
    if _load().oracle_attend(_ptr(q), Hq, d, _ptr(k), _ptr(v), T, float(c), _ptr(out), _ptr(lse)) != 0:
        raise MemoryError("oracle_attend: out of host memory")
    return out, lse


def merge_splits(outs, lses):
    """Attention over the union of disjoint parts of an attended set, from the parts.

    outs float64 [S][Hq][d] (each part's softmax-weighted mean of v), lses float64
    [S][Hq] (each part's log sum exp of the logits; -inf for an empty part).  For the
    softmax over the union, the log-sum-exp is log sum_j exp(lse_j) and the output is
    sum_j exp(lse_j - lse) * out_j: each part's exponentials summed over its own tokens
    are exp(lse_j), so its normalised output enters with weight exp(lse_j) / sum.
    Computed with the largest lse_j subtracted first.  All parts empty: out 0, lse -inf.
    """
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    S, Hq, d = outs.shape
    out = np.zeros((Hq, d))
    lse = np.full(Hq, -np.inf)
    for h in range(Hq):
        m = max(lses[j, h] for j in range(S))
        if m == -np.inf:
            continue
        wsum = 0.0
        for j in range(S):
            if lses[j, h] == -np.inf:
                continue
            wj = math.exp(lses[j, h] - m)
            wsum += wj
            out[h] += wj * outs[j, h]
        out[h] /= wsum
        lse[h] = m + math.log(wsum)
    return out, lse


# ---------------------------------------------------------------------------
# Attended sets
# ---------------------------------------------------------------------------

def attended_range(ctx_len: int, window: int):
    """Positions [lo, hi) a decode query attends; ctx_len includes the current token."""
    hi = int(ctx_len)
    lo = max(0, hi - int(window)) if window > 0 else 0
    return lo, hi


def prefill_ranges(prefix_len: int, n_new: int, window: int):
    """[lo, hi) per new token i: keys up to and including its own position p0+i."""
    out = []
    for i in range(n_new):
        hi = prefix_len + i + 1
        lo = max(0, hi - window) if window > 0 else 0
        out.append((lo, hi))
    return out


# ---------------------------------------------------------------------------
# Sequences: seeded fp32 K/V rows -> int8 codes and scales (logical, unpaged)
# ---------------------------------------------------------------------------

def seq_kv(seed: int, buffer: int, b: int, length: int, start: int = 0, dim: int = 128):
    """Codes and scales of K and V of sequence b in one buffer, positions start .. start+length-1."""
    kx = synth.kv_rows(seed, synth.stream_k(buffer), b, start, length, dim)
    vx = synth.kv_rows(seed, synth.stream_v(buffer), b, start, length, dim)
    kc, ks = quantize_rows(kx)
    vc, vs = quantize_rows(vx)
    return kc, ks, vc, vs


def query(bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> float64 (exact)."""
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def decode_seq(q_bits: np.ndarray, kc, ks, vc, vs, ctx_len: int, window: int, c: float):
    """Decode output of one sequence: q bits [Hq][d], logical codes/scales covering 0..ctx_len-1."""
    lo, hi = attended_range(ctx_len, window)
    k = dequantize(kc[lo:hi], ks[lo:hi])
    v = dequantize(vc[lo:hi], vs[lo:hi])
    return attend(query(q_bits), k, v, c)


def prefill_seq(q_bits: np.ndarray, kc, ks, vc, vs, prefix_len: int, window: int, c: float, tokens=None):
    """Prefill outputs of one sequence: q bits [n_new][Hq][d]; codes cover 0..prefix_len+n_new-1.

    Returns (out [len(tokens)][Hq][d], lse [len(tokens)][Hq]) for the new tokens listed (all by default).
    """
    n_new, Hq, d = q_bits.shape
    tokens = range(n_new) if tokens is None else tokens
    ranges = prefill_ranges(prefix_len, n_new, window)
    outs, lses = [], []
    for i in tokens:
        lo, hi = ranges[i]
        k = dequantize(kc[lo:hi], ks[lo:hi])
        v = dequantize(vc[lo:hi], vs[lo:hi])
        o, l = attend(query(q_bits[i]), k, v, c)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


# ---------------------------------------------------------------------------
# Paged pool layout
# ---------------------------------------------------------------------------

def page_bytes(page_size: int, head_dim: int = 128) -> int:
    return page_size * (2 * head_dim + 8)


def pool_new(num_pages: int, page_size: int, head_dim: int = 128, fill: int = 0xA5) -> np.ndarray:
    return np.full(num_pages * page_bytes(page_size, head_dim), fill, dtype=np.uint8)


def _page_views(pool: np.ndarray, page: int, P: int, d: int):
    base = page * page_bytes(P, d)
    kc = pool[base:base + P * d].view(np.int8).reshape(P, d)
    vc = pool[base + P * d:base + 2 * P * d].view(np.int8).reshape(d, P).T  # [slot][channel] view of [d][P]
    ks = pool[base + 2 * P * d:base + 2 * P * d + 4 * P].view(np.float32)
    vs = pool[base + 2 * P * d + 4 * P:base + 2 * P * d + 8 * P].view(np.float32)
    return kc, vc, ks, vs


def pool_write(pool: np.ndarray, table_row: np.ndarray, pos0: int, kc, ks, vc, vs, page_size: int,
               head_dim: int = 128) -> None:
    """Write tokens pos0 .. pos0+n-1 of one sequence into the pool through its block table row."""
    for j in range(kc.shape[0]):
        p = pos0 + j
        page = int(table_row[p // page_size])
        slot = p % page_size
        pkc, pvc, pks, pvs = _page_views(pool, page, page_size, head_dim)
        pkc[slot] = kc[j]
        pvc[slot] = vc[j]
        pks[slot] = ks[j]
        pvs[slot] = vs[j]


def pool_read(pool: np.ndarray, table_row: np.ndarray, length: int, page_size: int, head_dim: int = 128):
    """Walk a block table row and rebuild logical (kc, ks, vc, vs) for positions 0..length-1."""
    kc = np.empty((length, head_dim), dtype=np.int8)
    vc = np.empty((length, head_dim), dtype=np.int8)
    ks = np.empty(length, dtype=np.float32)
    vs = np.empty(length, dtype=np.float32)
    for p in range(length):
        pkc, pvc, pks, pvs = _page_views(pool, int(table_row[p // page_size]), page_size, head_dim)
        s = p % page_size
        kc[p], vc[p], ks[p], vs[p] = pkc[s], pvc[s], pks[s], pvs[s]
    return kc, ks, vc, vs


# ---------------------------------------------------------------------------
# KV-size formula
# ---------------------------------------------------------------------------

def kv_cache_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, dtype_bytes: float) -> float:
    """2 x layers x kv_heads x head_dim x bytes per value (K and V)."""
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes


def softmax_scale(head_dim: int = 128) -> float:
    return 1.0 / math.sqrt(head_dim)

"""Pins for the oracle: each check ties it to something other than itself
(closed forms, invariants, brute force at 50 digits, the pages' printed numbers)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

mpmath = pytest.importorskip("mpmath")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
C = 1.0 / math.sqrt(128.0)


# ---------------------------------------------------------------------------
# Quantizer (int8 KV cache: symmetric per-token absmax, fp32 scale, ties to even)
# ---------------------------------------------------------------------------

def test_quant_absmax_element_maps_to_127():
    x = synth.kv_rows(7, 0, 0, 0, 64)
    codes, scales = oracle.quantize_rows(x)
    for t in range(64):
        i = int(np.argmax(np.abs(x[t])))
        assert abs(int(codes[t, i])) == 127
        assert np.sign(codes[t, i]) == np.sign(x[t, i])
        assert scales[t] == np.float32(np.abs(x[t]).max()) / np.float32(127)


def test_quant_integer_inputs_are_exact():
    rng = np.random.default_rng(0)
    x = rng.integers(-127, 128, size=(32, 128)).astype(np.float32)
    x[:, 5] = 127.0  # amax 127 -> scale exactly 1
    codes, scales = oracle.quantize_rows(x)
    assert np.all(scales == 1.0)
    assert np.array_equal(codes.astype(np.float32), x)


def test_quant_ties_round_half_to_even():
    # With amax = 127 the scale is exactly 1, so x/s is x itself: halves are true ties.
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, 0] = 127.0
    halves = [0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5, -126.5]
    expect = [0, 2, 2, 4, 0, -2, -2, 126, -126]
    x[0, 1:1 + len(halves)] = halves
    codes, _ = oracle.quantize_rows(x)
    assert list(codes[0, 1:1 + len(halves)]) == expect


def test_quant_power_of_two_scaling_invariance():
    x = synth.kv_rows(11, 1, 3, 0, 32)
    c0, s0 = oracle.quantize_rows(x)
    for k in (-20, -3, 1, 9):
        c1, s1 = oracle.quantize_rows(x * np.float32(2.0 ** k))
        assert np.array_equal(c0, c1)
        assert np.array_equal(s1, s0 * np.float32(2.0 ** k))


def test_quant_zero_vector_and_error_bound():
    x = synth.kv_rows(13, 2, 1, 0, 256)
    x[3] = 0.0
    codes, scales = oracle.quantize_rows(x)
    assert scales[3] == 0.0 and not codes[3].any()
    assert codes.min() >= -127  # -128 is never produced
    err = np.abs(x.astype(np.float64) - scales[:, None].astype(np.float64) * codes)
    assert np.all(err <= scales[:, None] * (0.5 + 1e-5) + 0.0)


def test_quant_bruteforce_nearest_code():
    # Each code must be a nearest integer to the fp32 quotient x/s (ties checked above).
    x = synth.kv_rows(17, 3, 2, 0, 128)
    codes, scales = oracle.quantize_rows(x)
    ratio = x.astype(np.float64) / scales[:, None].astype(np.float64)
    assert np.all(np.abs(ratio - codes) <= 0.5 + 1e-5)


def _quant_division_rows():
    g = json.load(open(os.path.join(GOLDEN, "quant_division.json")))
    x = np.array([r["x_bits"] for r in g["rows"]], dtype=np.uint32).view(np.float32)
    codes = np.array([r["codes"] for r in g["rows"]], dtype=np.int64)
    scales = np.array([r["scale_bits"] for r in g["rows"]], dtype=np.uint32).view(np.float32)
    return g, x, codes, scales


def test_quant_division_golden():
    """Rows whose codes depend on the reading of the division: one IEEE fp32 division x/s
    and round half to even (values written from the definition with exact rationals)."""
    g, x, codes, scales = _quant_division_rows()
    assert g["case_counts"]["reciprocal"] >= 10 and g["case_counts"]["tie"] >= 10
    got_codes, got_scales = oracle.quantize_rows(x)
    assert np.array_equal(got_scales.view(np.uint32), scales.view(np.uint32))
    assert np.array_equal(got_codes.astype(np.int64), codes)


def _planted_quantizer(x, variant):
    """The oracle's quantizer with one plausible slip, on the CPU (numpy fp32)."""
    x = x.astype(np.float32)
    amax = np.abs(x).max(axis=1)
    s = (amax / np.float32(127)).astype(np.float32)
    if variant == "reciprocal":
        q = x * (np.float32(1) / s)[:, None]
    elif variant == "inverse_scale":
        q = x * (np.float32(127) / amax)[:, None]
    elif variant == "half_away":
        q = x / s[:, None]
        return np.clip(np.sign(q) * np.floor(np.abs(q) + np.float32(0.5)), -127, 127).astype(np.int64)
    else:
        q = x / s[:, None]
    return np.clip(np.rint(q.astype(np.float32)), -127, 127).astype(np.int64)


@pytest.mark.parametrize("variant", ["reciprocal", "inverse_scale", "half_away"])
def test_quant_division_golden_rejects_slips(variant):
    """Each slip gives other codes on the golden rows, so the golden test pins the reading."""
    _, x, codes, _ = _quant_division_rows()
    assert np.array_equal(_planted_quantizer(x, "plain"), codes)  # the plain numpy form agrees
    assert not np.array_equal(_planted_quantizer(x, variant), codes)


def test_quant_zero_scale_from_underflow():
    """amax / 127 below the smallest subnormal rounds the scale to 0: codes 0, like a zero vector."""
    x = np.zeros((4, 128), dtype=np.float32)
    tiny = np.float32(np.finfo(np.float32).smallest_subnormal)
    x[0, :4] = [tiny, -tiny, 2 * tiny, 0]            # amax/127 underflows to 0
    x[1, :2] = [np.float32(63) * tiny, -tiny]        # 63/127 of a subnormal still rounds to 0
    x[2, :2] = [np.float32(64) * tiny, -tiny]        # 64/127 rounds up: scale = smallest subnormal
    x[3, :2] = [np.float32(127) * tiny, -tiny]       # scale = smallest subnormal, codes exact
    codes, scales = oracle.quantize_rows(x)
    assert scales[0] == 0 and not codes[0].any()
    assert scales[1] == 0 and not codes[1].any()
    assert scales[2] == tiny and codes[2, 0] == 64 and codes[2, 1] == -1
    assert scales[3] == tiny and codes[3, 0] == 127 and codes[3, 1] == -1


# ---------------------------------------------------------------------------
# Attention (softmax over the attended tokens, one shared K/V head)
# ---------------------------------------------------------------------------

def _mp_attend(q, k, v, c):
    """Brute force at 50 digits: per-element sums and exps, no max trick."""
    mpmath.mp.dps = 50
    Hq, d = q.shape
    T = k.shape[0]
    out = np.zeros((Hq, d))
    lse = np.zeros(Hq)
    for h in range(Hq):
        z = [mpmath.mpf(c) * mpmath.fsum(mpmath.mpf(float(q[h, i])) * mpmath.mpf(float(k[t, i])) for i in range(d))
             for t in range(T)]
        w = [mpmath.exp(zt) for zt in z]
        s = mpmath.fsum(w)
        for i in range(d):
            out[h, i] = float(mpmath.fsum(w[t] * mpmath.mpf(float(v[t, i])) for t in range(T)) / s)
        lse[h] = float(mpmath.log(s))
    return out, lse


def _small_case(seed, T, Hq, d=128):
    kc, ks, vc, vs = oracle.seq_kv(seed, 0, 0, T)
    q = oracle.query(synth.q_rows(seed, synth.stream_q(0), 0, Hq))
    return q, oracle.dequantize(kc, ks), oracle.dequantize(vc, vs)


@pytest.mark.parametrize("T,Hq", [(1, 2), (2, 3), (4, 2), (7, 1)])
def test_attend_matches_50_digit_bruteforce(T, Hq):
    q, k, v = _small_case(100 + T, T, Hq)
    out, lse = oracle.attend(q, k, v, C)
    ref, ref_lse = _mp_attend(q, k, v, C)
    assert np.allclose(out, ref, atol=1e-13, rtol=0)
    assert np.allclose(lse, ref_lse, atol=1e-13, rtol=0)


def test_attend_single_token_returns_v():
    q, k, v = _small_case(3, 1, 4)
    out, lse = oracle.attend(q, k, v, C)
    assert np.array_equal(out, np.repeat(v, 4, axis=0))
    assert np.allclose(lse, C * (q @ k[0]), atol=1e-13)


def test_attend_two_tokens_closed_form():
    q, k, v = _small_case(5, 2, 3)
    out, _ = oracle.attend(q, k, v, C)
    for h in range(3):
        z0, z1 = C * q[h] @ k[0], C * q[h] @ k[1]
        s0 = 1.0 / (1.0 + math.exp(z1 - z0))
        assert np.allclose(out[h], s0 * v[0] + (1 - s0) * v[1], atol=1e-14)


def test_attend_identical_keys_give_mean_of_v():
    q, k, v = _small_case(9, 37, 4)
    k[:] = k[0]
    out, lse = oracle.attend(q, k, v, C)
    assert np.allclose(out, v.mean(axis=0)[None, :], atol=1e-13)
    assert np.allclose(lse, C * (q @ k[0]) + math.log(37), atol=1e-12)


def test_attend_key_shift_invariance():
    # Adding u to every key shifts each head's logits by c*q.u: outputs unchanged, lse shifted.
    q, k, v = _small_case(21, 50, 4)
    u = np.linspace(-1.0, 2.0, 128)
    out0, lse0 = oracle.attend(q, k, v, C)
    out1, lse1 = oracle.attend(q, k + u[None, :], v, C)
    assert np.allclose(out0, out1, atol=1e-12)
    assert np.allclose(lse1 - lse0, C * (q @ u), atol=1e-11)


def test_attend_token_permutation_and_head_independence():
    q, k, v = _small_case(23, 40, 5)
    out, lse = oracle.attend(q, k, v, C)
    perm = np.random.default_rng(1).permutation(40)
    out_p, lse_p = oracle.attend(q, k[perm], v[perm], C)
    assert np.allclose(out, out_p, atol=1e-13) and np.allclose(lse, lse_p, atol=1e-13)
    for h in range(5):
        o_h, l_h = oracle.attend(q[h:h + 1], k, v, C)
        assert np.array_equal(o_h[0], out[h]) and l_h[0] == lse[h]


def test_attend_empty_set():
    out, lse = oracle.attend(np.ones((2, 128)), np.zeros((0, 128)), np.zeros((0, 128)), C)
    assert not out.any() and np.all(np.isneginf(lse))


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_merge_splits_equals_unsplit(seed):
    """Cutting the attended set at any points (empty parts included) and merging the parts by
    their log-sum-exp gives the unsplit attention within 1e-12."""
    T, Hq = 300, 4
    q, k, v = _small_case(200 + seed, T, Hq)
    k *= 3.0  # a wide logit range, so the weights of the parts differ by many orders
    ref, ref_lse = oracle.attend(q, k, v, C)
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.integers(0, T + 1, size=int(rng.integers(1, 12))))
    edges = [0, *cuts.tolist(), T, T]  # repeated edges give empty parts
    parts = [oracle.attend(q, k[a:b], v[a:b], C) for a, b in zip(edges[:-1], edges[1:])]
    assert any(b == a for a, b in zip(edges[:-1], edges[1:]))
    out, lse = oracle.merge_splits([o for o, _ in parts], [l for _, l in parts])
    assert np.abs(out - ref).max() <= 1e-12
    assert np.abs(lse - ref_lse).max() <= 1e-12


def test_merge_splits_single_part_and_all_empty():
    q, k, v = _small_case(301, 20, 3)
    o, l = oracle.attend(q, k, v, C)
    out, lse = oracle.merge_splits([o], [l])
    assert np.array_equal(out, o) and np.allclose(lse, l, atol=0, rtol=1e-15)
    e_o, e_l = oracle.attend(q, k[:0], v[:0], C)
    out, lse = oracle.merge_splits([e_o, e_o], [e_l, e_l])
    assert not out.any() and np.all(np.isneginf(lse))


def _position_coded_values(L):
    # q = 0 makes attention the plain mean over the attended set; V rows carry their position.
    v = np.repeat(np.arange(L, dtype=np.float64)[:, None], 128, axis=1)
    return np.zeros((2, 128)), np.zeros((L, 128)), v


@pytest.mark.parametrize("L,W", [(1, 1024), (1000, 1024), (1024, 1024), (1025, 1024), (5000, 1024), (5000, 0),
                                 (300, 16)])
def test_decode_window_is_last_W_positions(L, W):
    q, k, v = _position_coded_values(L)
    lo, hi = oracle.attended_range(L, W)
    out, lse = oracle.attend(q, k[lo:hi], v[lo:hi], C)
    n = min(L, W) if W else L
    assert hi == L and hi - lo == n
    assert np.allclose(out, (L - 1 + L - n) / 2.0, atol=1e-9)
    assert np.allclose(lse, math.log(n), atol=1e-12)


def test_window_at_least_context_equals_global():
    kc, ks, vc, vs = oracle.seq_kv(31, 0, 0, 700)
    qb = synth.q_rows(31, synth.stream_q(0), 0, 4)
    g = oracle.decode_seq(qb, kc, ks, vc, vs, 700, 0, C)
    w = oracle.decode_seq(qb, kc, ks, vc, vs, 700, 700, C)
    w2 = oracle.decode_seq(qb, kc, ks, vc, vs, 700, 4096, C)
    assert np.array_equal(g[0], w[0]) and np.array_equal(g[0], w2[0])


def test_prefill_ranges_causal_and_position_coded():
    p0, n = 40, 9
    ranges = oracle.prefill_ranges(p0, n, 0)
    assert ranges == [(0, p0 + i + 1) for i in range(n)]
    q, k, v = _position_coded_values(p0 + n)
    for i, (lo, hi) in enumerate(ranges):
        out, _ = oracle.attend(q, k[lo:hi], v[lo:hi], C)
        assert np.allclose(out, (p0 + i) / 2.0, atol=1e-9)  # mean of 0..p0+i
    assert oracle.prefill_ranges(p0, 3, 16) == [(25, 41), (26, 42), (27, 43)]


def test_prefill_last_token_equals_decode():
    # Prefix reuse: the last new token of a chunk sees exactly what a decode step at that length sees.
    kc, ks, vc, vs = oracle.seq_kv(41, 0, 0, 300)
    qb = synth.q_rows(41, synth.stream_q(0), 0, 5 * 4).reshape(5, 4, 128)
    out, lse = oracle.prefill_seq(qb, kc, ks, vc, vs, 295, 0, C)
    d_out, d_lse = oracle.decode_seq(qb[4], kc, ks, vc, vs, 300, 0, C)
    assert np.array_equal(out[4], d_out) and np.array_equal(lse[4], d_lse)


def test_shared_buffer_equals_duplicated_buffer():
    # Layers that share one KV buffer see the same bytes as layers given a private copy of it.
    kc, ks, vc, vs = oracle.seq_kv(43, 0, 2, 400)
    qb = synth.q_rows(43, synth.stream_q(1), 2, 4)
    shared = oracle.decode_seq(qb, kc, ks, vc, vs, 400, 128, C)
    dup = oracle.decode_seq(qb, kc.copy(), ks.copy(), vc.copy(), vs.copy(), 400, 128, C)
    assert np.array_equal(shared[0], dup[0])


# ---------------------------------------------------------------------------
# Paged layout
# ---------------------------------------------------------------------------

def test_pool_layout_byte_offsets_by_hand():
    P, d = 16, 128
    assert oracle.page_bytes(P, d) == 16 * 264 == 4224
    pool = oracle.pool_new(8, P, d, fill=0)
    table = np.array([5, 2, 7], dtype=np.int32)
    kc = np.full((1, d), 3, dtype=np.int8)
    vc = np.full((1, d), -4, dtype=np.int8)
    oracle.pool_write(pool, table, 17, kc, np.array([0.25], np.float32), vc, np.array([0.5], np.float32), P, d)
    base = 2 * 4224  # position 17 -> table[1] = page 2, slot 1
    assert np.all(pool[base + 128:base + 256] == 3)  # K: token-major, slot 1 = bytes 128..255
    v_block = pool[base + 2048:base + 4096].view(np.int8).reshape(128, 16)  # V: channel-major [d][P]
    assert np.all(v_block[:, 1] == -4) and np.count_nonzero(v_block) == 128
    assert pool[base + 4096 + 4:base + 4096 + 8].view(np.float32)[0] == 0.25
    assert pool[base + 4096 + 64 + 4:base + 4096 + 64 + 8].view(np.float32)[0] == 0.5
    float_bytes = np.count_nonzero(np.array([0.25, 0.5], np.float32).view(np.uint8))
    assert np.count_nonzero(pool) == 128 + 128 + float_bytes  # nothing else touched


def test_pool_roundtrip_random_table():
    P, d, L = 16, 128, 77
    table, npages = synth.block_table(5, 9, np.array([L]), P, 8)
    pool = oracle.pool_new(npages, P, d)
    kc, ks, vc, vs = oracle.seq_kv(5, 0, 0, L)
    oracle.pool_write(pool, table[0], 0, kc, ks, vc, vs, P, d)
    r = oracle.pool_read(pool, table[0], L, P, d)
    for a, b in zip(r, (kc, ks, vc, vs)):
        assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# KV-size formula against the page's worked numbers
# ---------------------------------------------------------------------------

def test_kv_size_formula_matches_page_examples():
    g = json.load(open(os.path.join(GOLDEN, "kv_size_examples.json")))
    for case in g["cases"]:
        per_tok = oracle.kv_cache_bytes_per_token(case["layers"], case["kv_heads"], case["head_dim"], case["bytes"])
        got = per_tok * case["layer_fraction"] * case["tokens"]
        assert abs(got / case["page_value_bytes"] - 1.0) <= g["rel_tol"], case["what"]
    dense = oracle.kv_cache_bytes_per_token(80, 8, 128, 2)
    eff = oracle.kv_cache_bytes_per_token(36, 8, 64, 2) * 0.5
    assert abs(dense / eff / g["ratio"]["page_value"] - 1.0) <= g["ratio"]["rel_tol"]

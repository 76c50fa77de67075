"""Seeded generators: determinism, distribution and bf16 rounding."""
import numpy as np

import synth


def test_normal_moments_and_grid():
    x = synth.kv_rows(1234, 0, 5, 100, 2000)
    assert x.dtype == np.float32 and x.shape == (2000, 128)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.var()) - 1.0) < 0.02
    assert np.all(np.abs(x) < 6.0)
    assert np.all((x * (1 << 20)) == np.rint(x * (1 << 20)))  # multiples of 2^-20


def test_counters_are_positional():
    a = synth.kv_rows(9, 3, 7, 10, 20)
    b = synth.kv_rows(9, 3, 7, 15, 10)
    assert np.array_equal(a[5:15], b)
    assert not np.array_equal(synth.kv_rows(9, 4, 7, 10, 20), a)
    assert not np.array_equal(synth.kv_rows(10, 3, 7, 10, 20), a)


def test_splitmix64_reference_values():
    # Published splitmix64 with seed 1234567: first outputs of the reference stream.
    out = synth.splitmix64(1234567, np.arange(5, dtype=np.uint64))
    expect = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
              16408922859458223821]
    assert [int(v) for v in out] == expect


def test_bf16_rne():
    one = np.float32(1.0)
    vals = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -2.5, 3.0e38], dtype=np.float32)
    bits = synth.bf16_bits_rne(vals)
    back = synth.bf16_bits_to_f32(bits)
    assert back[0] == one
    assert back[1] == one                       # tie -> even (1.0)
    assert back[2] == np.float32(1.0 + 4 * 2.0 ** -8)  # tie -> even (1 + 2^-6)
    assert back[3] == one
    assert back[4] == np.float32(-2.5)
    assert np.isfinite(back[5])


def test_block_table_is_a_partial_permutation():
    L = synth.uniform_int(3, 1, 50, 10, 300)
    table, n = synth.block_table(3, 7, L, 16, 19)
    used = table[table >= 0]
    assert len(used) == n == sum((int(l) + 15) // 16 for l in L)
    assert len(np.unique(used)) == len(used) and used.min() == 0 and used.max() == n - 1


def test_workloads():
    for c in (1, 2, 3, 4, 5):
        w = synth.workload(c)
        assert len(w.ctx_len) == w.batch
    w = synth.workload(3)
    assert w.layer_to_buffer == [0, 0, 1, 1, 2, 3] and w.layer_windows == [1024] * 5 + [0]
    assert w.ctx_len.min() >= 256 and w.ctx_len.max() <= 32768
    assert 3500 < np.median(w.ctx_len) < 4700

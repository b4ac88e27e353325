"""The seeded input generator: its published random source and the workload
recipes (shapes, ranges, structure).  CPU only."""
import numpy as np

import dsa_inputs as gen


def test_splitmix64_matches_published_output():
    # SplitMix64 (Steele, Lea, Flood 2014) started from state 1234567: the first
    # five outputs of the reference implementation.
    z = gen._draws_chunk(1234567, 0, 5)
    assert [int(v) for v in z] == [6457827717110365317, 3203168211198807973,
                                   9817491932198370423, 4593380528125082431,
                                   16408922859458223821]


def test_counter_streams_are_position_independent_and_deterministic():
    a = gen.draws(7, 3, 10_000_000)
    b = gen.draws(7, 3, 100, start=5_000_000)
    assert np.array_equal(a[5_000_000:5_000_100], b)
    assert np.array_equal(gen.draws(7, 3, 50), a[:50])
    assert not np.array_equal(gen.draws(7, 4, 50), a[:50])


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    got = gen.bf16_bits_to_f64(gen.f32_to_bf16_bits(x))
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0 + 2 ** -7]


def test_distributions():
    v = gen.uniform_nibbles(1, 1, 1_600_000)
    assert v.min() == -8 and v.max() == 7
    cnt = np.bincount(v.astype(np.int64) + 8)
    assert abs(cnt / len(v) - 1 / 16).max() < 2e-3
    w = gen.uniform_int(1, 2, 100_000, 1, 4)
    assert set(np.unique(w).tolist()) == {1, 2, 3, 4}
    z = gen.bf16_bits_to_f64(gen.normal_bf16(1, 3, 400_000))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs((np.abs(z) < 1).mean() - 0.6827) < 0.005


def test_workload_shapes_and_structure():
    t = gen.tiny()
    assert (t.R, t.L_total, t.H_i, t.D_i, t.k, t.H_q, t.D_k, t.D_v) == (1, 4096, 4, 32, 256, 8, 64, 64)
    q = gen.bf16_bits_to_f64(t.q)
    assert abs(q.std() - 0.125) < 0.01
    x = gen.l64k(L=20000)
    assert x.k_idx.shape == (20000, 128) and x.q_idx.shape == (1, 64, 128)
    assert x.k_idx.min() >= -10 and x.k_idx.max() <= 9
    near = (np.abs(x.k_idx.astype(int) - x.q_idx[0, 0].astype(int)[None]) <= 2).all(1)
    assert 0.09 < near.mean() < 0.11
    c = gen.causal64(L=1000, R=64)
    assert c.row_len.tolist() == list(range(937, 1001))
    assert len(np.unique(c.k_idx, axis=0)) == 16
    b = gen.batch32()
    lens = np.diff(b.offsets)
    assert b.B == 32 and lens.min() >= 4096 and lens.max() <= 131072
    assert b.row_len.tolist() == lens.tolist()
    p = gen.prefill(L=3000, R=512)
    assert (p.R, p.B, p.L_total) == (512, 1, 3000)
    assert p.row_len.tolist() == list(range(2489, 3001))
    assert p.row_offsets.tolist() == [0, 512] and p.kv_format == "bf16" and p.kv_scale is None
    near = (np.abs(p.k_idx.astype(int) - p.q_idx[0, 0].astype(int)[None]) <= 2).all(1)
    assert 0.08 < near.mean() < 0.12


def test_fp8_cache_keeps_everything_but_the_cache():
    x = gen.l64k(L=700)
    y = gen.fp8_cache(x)
    for f in ("q_idx", "w_idx", "k_idx", "q", "offsets", "row_offsets", "row_len"):
        assert np.array_equal(getattr(x, f), getattr(y, f)), f
    assert y.kv.dtype == np.uint8 and y.kv_scale.dtype == np.float32 and y.kv_scale.shape == (700,)
    assert (y.kv_scale > 0).all() and x.kv_format == "bf16"
    # deterministic: the same problem gives the same codes
    assert np.array_equal(gen.fp8_cache(gen.l64k(L=700)).kv, y.kv)

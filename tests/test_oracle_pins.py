"""Pins for the CPU oracle, against facts that do not come from the oracle itself:
a hand-worked example, closed forms, special cases that reduce to a library
routine, and the properties that define an ordered top-k.  CPU only."""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import dsa_inputs as gen
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read_hand():
    rows = {}
    with open(os.path.join(GOLD, "indexer_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append([int(v) for v in vals])
    return rows


def _single(q_idx, w, k_idx, row_len=None):
    k_idx = np.asarray(k_idx, np.int8)
    L = k_idx.shape[0]
    return (np.asarray(q_idx, np.int8)[None], np.asarray(w, np.int32)[None],
            np.asarray(k_idx, np.int8), np.array([0, L], np.int32), np.array([0, 1], np.int32),
            np.array([L if row_len is None else row_len], np.int32))


# ---------------------------------------------------------------- scores

def test_scores_hand_worked_example():
    h = _read_hand()
    args = _single(h["q"], h["w"][0], h["k"])
    s = oracle.indexer_scores(*args)[0]
    assert s.tolist() == h["scores"][0]
    s2 = oracle.indexer_scores(*args, relu=False)[0]
    assert s2.tolist() == h["scores_norelu"][0]
    assert oracle.topk_indices(s, 2).tolist() == h["top2"][0]


def test_scores_without_relu_equal_weighted_query_closed_form():
    # Without the ReLU the head sum is linear: s = (sum_h w_h q_h) . k.
    x = gen.l64k(L=777)
    s = oracle.indexer_scores(x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len,
                              relu=False)[0]
    qbar = (x.w_idx[0].astype(np.int64)[:, None] * x.q_idx[0].astype(np.int64)).sum(0)
    assert np.array_equal(s, x.k_idx.astype(np.int64) @ qbar)


def test_scores_one_hot_queries_select_key_columns():
    # q_h = c_h * e_{j_h}: each head's dot is c_h * k[t, j_h]; catches a transposed
    # operand or a head/dim index mix-up.
    rng = np.random.default_rng(5)
    H, D, L = 6, 32, 50
    j = rng.choice(D, H, replace=False)
    c = rng.integers(-3, 4, H)
    q = np.zeros((H, D), np.int8)
    q[np.arange(H), j] = c
    w = rng.integers(1, 5, H)
    k = rng.integers(-128, 128, (L, D)).astype(np.int8)
    s = oracle.indexer_scores(*_single(q, w, k))[0]
    expect = np.zeros(L, np.int64)
    for h in range(H):
        expect += int(w[h]) * np.maximum(0, int(c[h]) * k[:, j[h]].astype(np.int64))
    assert np.array_equal(s, expect)


def test_scores_relu_invariants_and_head_permutation():
    x = gen.tiny(L=500)
    args = (x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len)
    s = oracle.indexer_scores(*args)[0]
    s_lin = oracle.indexer_scores(*args, relu=False)[0]
    assert (s >= 0).all() and (s >= s_lin).all()        # w >= 1 and relu(x) >= x
    perm = np.array([2, 0, 3, 1])
    s_p = oracle.indexer_scores(x.q_idx[:, perm], x.w_idx[:, perm], *args[2:])[0]
    assert np.array_equal(s, s_p)
    # doubling the weights doubles every score
    s2 = oracle.indexer_scores(x.q_idx, 2 * x.w_idx, *args[2:])[0]
    assert np.array_equal(s2, 2 * s)


def test_scores_antiparallel_single_head_is_zero():
    k = np.array([[3, -2, 5, 1], [1, 1, 1, 1]], np.int8)
    q = -k[0:1]
    s = oracle.indexer_scores(*_single(q, [7], k))[0]
    assert s[0] == 0 and s[1] == 7 * max(0, int(-(k[0].astype(int) @ k[1].astype(int))))


def test_scores_varlen_uses_each_request_and_row_length():
    x = gen.batch32(B=3, lo=40, hi=90)
    s = oracle.indexer_scores(x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len)
    for b in range(3):
        lo, hi = x.offsets[b], x.offsets[b + 1]
        alone = oracle.indexer_scores(*_single(x.q_idx[b], x.w_idx[b], x.k_idx[lo:hi]))[0]
        assert np.array_equal(s[b], alone)
    # a shorter visible length truncates, and what lies past it does not matter
    kk = x.k_idx.copy()
    rl = x.row_len.copy()
    rl[1] -= 7
    kk[x.offsets[1] + rl[1]:x.offsets[2]] = 127
    s2 = oracle.indexer_scores(x.q_idx, x.w_idx, kk, x.offsets, x.row_offsets, rl)
    assert np.array_equal(s2[1], s[1][:rl[1]])


def test_scores_causal_rows_share_one_cache():
    x = gen.causal64(L=300, R=5)
    s = oracle.indexer_scores(x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len)
    assert [len(v) for v in s] == [296, 297, 298, 299, 300]
    for r in range(5):
        alone = oracle.indexer_scores(*_single(x.q_idx[r], x.w_idx[r], x.k_idx))[0]
        assert np.array_equal(s[r], alone[:len(s[r])])


def test_scores_overflow_is_detected():
    k = np.full((2, 32), -128, np.int8)
    q = np.full((4, 32), -128, np.int8)
    with pytest.raises(OverflowError):
        oracle.indexer_scores(*_single(q, [1 << 20] * 4, k))


# ---------------------------------------------------------------- top-k

def _check_topk_definition(s, k, idx):
    """The properties that define the ordered top-k uniquely."""
    s = np.asarray(s)
    n = len(s)
    m = min(k, n)
    assert len(idx) == k
    assert (idx[m:] == -1).all()
    sel = idx[:m]
    assert len(set(sel.tolist())) == m and ((sel >= 0) & (sel < n)).all()
    # order: score descending, index ascending among equals
    for a, b in zip(sel[:-1], sel[1:]):
        assert s[a] > s[b] or (s[a] == s[b] and a < b)
    # dominance: every unselected position loses to every selected one
    chosen = np.zeros(n, bool)
    chosen[sel] = True
    for u in np.nonzero(~chosen)[0]:
        for v in sel:
            assert s[v] > s[u] or (s[v] == s[u] and v < u)


def test_topk_hand_example():
    s = [3, 1, 3, 2, 1, 0]
    assert oracle.topk_indices(s, 4).tolist() == [0, 2, 3, 1]
    assert oracle.topk_indices(s, 10).tolist() == [0, 2, 3, 1, 4, 5, -1, -1, -1, -1]
    assert oracle.topk_indices([], 3).tolist() == [-1, -1, -1]
    assert oracle.topk_indices([-5, oracle.INT32_MIN, oracle.INT32_MAX], 2).tolist() == [2, 0]


def test_topk_exhaustive_small_against_definition():
    for n in range(0, 7):
        for s in itertools.product(range(3), repeat=n):
            for k in range(1, n + 3):
                _check_topk_definition(s, k, oracle.topk_indices(s, k))


def test_topk_permutation_of_unique_scores():
    rng = np.random.default_rng(1)
    s = rng.permutation(10_000)[:3000] - 5000
    perm = rng.permutation(3000)
    a = oracle.topk_indices(s, 100)
    b = oracle.topk_indices(s[perm], 100)
    assert np.array_equal(s[a], s[perm][b])               # same score sequence
    assert np.array_equal(perm[b], a)                     # same positions, renamed


def test_topk_heavy_ties_take_lowest_indices():
    x = gen.causal64(L=4000, R=2, k=300)
    s = oracle.indexer_scores(x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len)[0]
    idx = oracle.topk_indices(s, 300)
    T = s[idx[-1]]
    ties = np.nonzero(s == T)[0]
    taken = idx[s[idx] == T]
    assert len(ties) > len(taken) > 0                      # the threshold is ambiguous
    assert np.array_equal(taken, ties[:len(taken)])
    _check_fast(s, 300, idx)


def _check_fast(s, k, idx):
    s = np.asarray(s)
    m = min(k, len(s))
    sel = idx[:m]
    ss = s[sel]
    assert (np.diff(ss) <= 0).all()
    eq = np.diff(ss) == 0
    assert (np.diff(sel)[eq] > 0).all()
    rest = np.ones(len(s), bool)
    rest[sel] = False
    if m and rest.any():
        T = ss[-1]
        assert s[rest].max() <= T
        assert (np.nonzero(rest & (s == T))[0] > sel[ss == T].max()).all()


def test_topk_l_le_k_selects_all_in_order():
    x = gen.tiny(L=200)
    s = oracle.indexer_scores(x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len)[0]
    idx = oracle.topk_indices(s, 256)
    assert sorted(idx[:200].tolist()) == list(range(200)) and (idx[200:] == -1).all()
    _check_fast(s, 256, idx)


# ---------------------------------------------------------------- attention

def _bf16(x):
    return gen.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_attention_single_selected_row_returns_its_value():
    x = gen.tiny(L=64)
    o = oracle.sparse_attention(x.q[0], x.kv, np.array([17, -1, -1]), x.D_v, 1.0)
    v = gen.bf16_bits_to_f64(x.kv[17, :x.D_v])
    assert np.array_equal(o, np.broadcast_to(v, o.shape))


def test_attention_zero_query_gives_mean_of_values():
    x = gen.l64k(L=300)
    q = np.zeros_like(x.q[0])
    idx = np.array([5, 99, 250, 3])
    o = oracle.sparse_attention(q, x.kv, idx, 512, 1 / 24)
    v = gen.bf16_bits_to_f64(x.kv[idx, :512]).mean(0)
    np.testing.assert_allclose(o, np.broadcast_to(v, o.shape), rtol=0, atol=1e-15)


def test_attention_two_rows_logistic_closed_form_uses_rope_columns():
    # Rows differ only in the rope columns (c >= D_v): the logit gap comes from
    # there alone, so a key restricted to D_v columns would give weights 1/2.
    D_k, D_v = 576, 512
    kv = np.zeros((2, D_k), np.float32)
    kv[:, :D_v] = np.array([[1.0], [-2.0]]) * np.linspace(-1, 1, D_v)[None]
    kv[0, 512] = 2.0
    kv[1, 513] = 0.5
    q = np.zeros((3, D_k), np.float32)
    q[0, 512] = 1.0
    q[1, 513] = 4.0
    q[2, 512], q[2, 513] = 0.25, -1.0
    scale = 0.5
    o = oracle.sparse_attention(_bf16(q), _bf16(kv), np.array([0, 1]), D_v, scale)
    V = gen.bf16_bits_to_f64(_bf16(kv))[:, :D_v]
    for h, gap in enumerate([scale * 2.0, scale * (0 - 2.0), scale * (0.5 + 0.5)]):
        p0 = 1.0 / (1.0 + math.exp(-gap))
        np.testing.assert_allclose(o[h], p0 * V[0] + (1 - p0) * V[1], rtol=0, atol=1e-14)


def test_attention_one_hot_rows_reduce_to_textbook_softmax():
    rng = np.random.default_rng(3)
    D_k, D_v, n = 64, 64, 9
    cols = rng.choice(D_v, n, replace=False)
    a = rng.choice([0.5, 1.0, 2.0], n)
    kv = np.zeros((n, D_k), np.float32)
    kv[np.arange(n), cols] = a
    q = rng.standard_normal((4, D_k)).astype(np.float32)
    qb, kvb = _bf16(q), _bf16(kv)
    Q = gen.bf16_bits_to_f64(qb)
    scale = 0.25
    o = oracle.sparse_attention(qb, kvb, np.arange(n), D_v, scale)
    p = sp_softmax(scale * Q[:, cols] * a[None, :], axis=1)
    np.testing.assert_allclose(o[:, cols], p * a[None, :], rtol=1e-13, atol=1e-15)
    mask = np.ones(D_v, bool)
    mask[cols] = False
    assert (o[:, mask] == 0).all()


def test_attention_is_invariant_to_selection_order():
    x = gen.l64k(L=3000)
    rng = np.random.default_rng(9)
    idx = rng.choice(3000, 700, replace=False)
    o1 = oracle.sparse_attention(x.q[0], x.kv, idx, 512, 1 / 24)
    o2 = oracle.sparse_attention(x.q[0], x.kv, rng.permutation(idx), 512, 1 / 24)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_decode_step_with_k_ge_L_is_dense_softmax_attention():
    x = gen.make_inputs("t", seed=11, lengths=[150], H_i=4, D_i=32, H_q=8, D_k=96, D_v=64,
                        k=256, softmax_scale=0.125)
    _, idx, out = oracle.decode_step(x)
    assert sorted(idx[0, :150].tolist()) == list(range(150))
    Q = gen.bf16_bits_to_f64(x.q[0])
    K = gen.bf16_bits_to_f64(x.kv)
    dense = sp_softmax(0.125 * Q @ K.T, axis=1) @ K[:, :64]
    np.testing.assert_allclose(out[0], dense, rtol=0, atol=1e-12)


def test_attention_scale_equals_scaled_query():
    x = gen.tiny(L=100)
    idx = np.arange(0, 100, 3)
    q2 = _bf16(gen.bf16_bits_to_f64(x.q[0]).astype(np.float32) * 2.0)   # exact (power of two)
    a = oracle.sparse_attention(x.q[0], x.kv, idx, 64, 2.0)
    b = oracle.sparse_attention(q2, x.kv, idx, 64, 1.0)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_attention_no_selection_is_zero():
    x = gen.tiny(L=10)
    o = oracle.sparse_attention(x.q[0], x.kv, np.full(4, -1), 64, 1.0)
    assert o.shape == (8, 64) and not o.any()


def test_attention_lse_closed_forms():
    # one row: the lse is its own logit; two rows: log(e^a + e^b)
    D = 64
    kv = np.zeros((2, D), np.float32)
    kv[0, 3] = 2.0
    kv[1, 5] = 1.0
    q = np.zeros((1, D), np.float32)
    q[0, 3], q[0, 5] = 0.5, -1.5
    qb, kvb = _bf16(q), _bf16(kv)
    a, b = 0.25 * 0.5 * 2.0, 0.25 * -1.5 * 1.0
    assert oracle.attention_lse(qb, kvb, np.array([0]), 0.25)[0] == a
    np.testing.assert_allclose(oracle.attention_lse(qb, kvb, np.array([0, 1]), 0.25)[0],
                               math.log(math.exp(a) + math.exp(b)), rtol=1e-15)
    assert oracle.attention_lse(qb, kvb, np.array([-1]), 0.25)[0] == -np.inf


# ---------------------------------------------------------------- FP8 cache

def test_e4m3_decode_matches_library_for_all_codes():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    a = oracle.e4m3_to_f64(codes)
    b = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(a), np.isnan(b))
    ok = ~np.isnan(a)
    assert np.array_equal(a[ok], b[ok]) and np.array_equal(np.signbit(a[ok]), np.signbit(b[ok]))


def test_e4m3_decode_named_values():
    # OCP E4M3: bias 7, subnormals at E = 0, S.1111.111 NaN, max 448.
    named = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0 ** -6, 0x07: 7 * 2.0 ** -9, 0x01: 2.0 ** -9, 0x81: -(2.0 ** -9),
             0x77: 240.0, 0x78: 256.0}
    got = oracle.e4m3_to_f64(np.array(list(named), np.uint8))
    assert got.tolist() == list(named.values())
    assert np.signbit(oracle.e4m3_to_f64(np.array([0x80], np.uint8))[0])
    assert np.isnan(oracle.e4m3_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()
    # every finite non-NaN code is distinct and ordered within each sign
    pos = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    assert (np.diff(pos) > 0).all()


def _fp8_codes(vals):
    import torch
    return torch.tensor(np.asarray(vals, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_fp8_attention_two_rows_logistic_closed_form_with_scales():
    # Row j is worth s_j * code_j: the scale must reach the logit and the value.
    D = 32
    c = np.zeros((2, D), np.float32)
    c[0, 0], c[0, 1] = 2.0, 1.5
    c[1, 0], c[1, 2] = -1.0, 3.0
    codes = _fp8_codes(c)
    s = np.array([0.3, 1.7], np.float32)
    q = np.zeros((2, D), np.float32)
    q[0, 0] = 1.0
    q[1, 1], q[1, 2] = 0.5, -0.25
    qb = _bf16(q)
    scale = 0.75
    o = oracle.sparse_attention(qb, codes, np.array([0, 1]), D, scale, kv_scale_req=s)
    V = c.astype(np.float64) * s.astype(np.float64)[:, None]
    Q = gen.bf16_bits_to_f64(qb)
    for h in range(2):
        z = scale * (Q[h] @ V.T)
        p0 = 1.0 / (1.0 + math.exp(z[1] - z[0]))
        np.testing.assert_allclose(o[h], p0 * V[0] + (1 - p0) * V[1], rtol=0, atol=1e-14)
    lse = oracle.attention_lse(qb, codes, np.array([0, 1]), scale, kv_scale_req=s)
    z = scale * (Q @ V.T)
    np.testing.assert_allclose(lse, np.log(np.exp(z).sum(1)), rtol=1e-14)


def test_fp8_attention_with_power_of_two_scales_equals_bf16_rows():
    # s_j = 2^e_j: s_j * e4m3(code) is a bf16 value, so the FP8 problem is the
    # bf16 problem over rows that the library's own conversion produces.
    import torch
    x = gen.fp8_cache(gen.l64k(L=400))
    rng = np.random.default_rng(5)
    s = np.exp2(rng.integers(-3, 3, x.L_total)).astype(np.float32)
    rows = torch.from_numpy(x.kv).view(torch.float8_e4m3fn).to(torch.bfloat16)
    rows = (rows * torch.from_numpy(s).to(torch.bfloat16)[:, None]).view(torch.int16).numpy().view(np.uint16)
    idx = rng.choice(400, 150, replace=False)
    a = oracle.sparse_attention(x.q[0], x.kv, idx, 512, 1 / 24, kv_scale_req=s)
    b = oracle.sparse_attention(x.q[0], rows, idx, 512, 1 / 24)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    c = oracle.sparse_attention(x.q[0], x.kv, idx, 512, 1 / 24)          # scales dropped
    assert np.abs(a - c).max() > 1e-3


def test_fp8_cache_writer_round_trip_is_within_half_an_e4m3_step():
    x = gen.l64k(L=500)
    y = gen.fp8_cache(x)
    assert y.kv.dtype == np.uint8 and y.kv.shape == x.kv.shape and y.kv_format == "e4m3"
    assert not np.isin(y.kv, [0x7F, 0xFF]).any()
    ref = gen.bf16_bits_to_f64(x.kv)
    sc = y.kv_scale.astype(np.float64)[:, None]
    back = oracle.e4m3_to_f64(y.kv) * sc
    # relative half step 2^-4 for normals, absolute half of the subnormal step
    assert (np.abs(back - ref) <= np.maximum(np.abs(ref) * 2.0 ** -4, sc * 2.0 ** -10) * 1.0001).all()
    # each row's largest magnitude lands on the largest code
    assert (np.abs(oracle.e4m3_to_f64(y.kv)).max(1) == 448.0).all()
    z = gen.fp8_cache(x, with_scale=False)
    assert z.kv_scale is None
    np.testing.assert_allclose(oracle.e4m3_to_f64(z.kv), ref, rtol=2.0 ** -4, atol=2.0 ** -10)


def test_fp8_decode_step_uses_the_scales():
    x = gen.fp8_cache(gen.tiny(L=600))
    _, idx, out = oracle.decode_step(x)
    rows = oracle.e4m3_to_f64(x.kv) * x.kv_scale.astype(np.float64)[:, None]
    sel = idx[0][idx[0] >= 0]
    z = x.softmax_scale * (gen.bf16_bits_to_f64(x.q[0]) @ rows[sel].T)
    np.testing.assert_allclose(out[0], sp_softmax(z, axis=1) @ rows[sel, :x.D_v], rtol=0, atol=1e-13)

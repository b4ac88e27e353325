"""The tcgen05 tensor-core indexer: bit-exact scores against the CPU oracle and
against the dp4a indexer, over the shapes and layouts it serves (one row per
request, causal row groups of up to four rows, packed varlen caches, ragged
tiles, extreme int8 values, the linear variant, 32/64/128 heads, D_i 64/128)."""
import numpy as np
import pytest

import dsa_inputs as gen
import oracle
from gpu_harness import value_bound

pytestmark = pytest.mark.gpu


def _scores(x, indexer, relu=True, qk=0):
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    prob, t = dsa.upload_inputs(x, indexer=indexer, relu=relu, qk_abs_max=qk)
    assert dsa.indexer_kind(prob) == indexer
    ws = dsa.alloc_workspace(prob)
    s = torch.full((x.R, max(1, x.L_max)), -99, dtype=torch.int32, device="cuda")
    dsa.dsa_index_scores(prob, s, ws)
    status = dsa.dsa_read_device_status(ws)
    return s.cpu().numpy(), status


def _check(x, rows=None, relu=True, vs_dp4a=True):
    """Both conversions: exact (no declared bound) and biased (declared bound)."""
    for qk in (0, value_bound(x)):
        _check_one(x, rows, relu, vs_dp4a, qk)


def _check_one(x, rows, relu, vs_dp4a, qk):
    got, status = _scores(x, "tc", relu, qk)
    assert status == 0
    rows = list(range(x.R)) if rows is None else rows
    ref = oracle.indexer_scores(x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len,
                                relu=relu, rows=rows)
    for j, r in enumerate(rows):
        n = int(x.row_len[r])
        assert np.array_equal(got[r, :n], ref[j]), f"row {r}"
        assert (got[r, n:] == -99).all(), f"row {r}: wrote past its length"
    if vs_dp4a:
        other, _ = _scores(x, "dp4a", relu)
        for r in range(x.R):
            n = int(x.row_len[r])
            assert np.array_equal(got[r, :n], other[r, :n])


def test_tc_small_single_row():
    _check(gen.l64k(L=1000))


@pytest.mark.parametrize("L", [1, 127, 128, 129, 4099, 65536])
def test_tc_lengths(L):
    _check(gen.l64k(L=L))


def test_tc_long_context_layer():
    _check(gen.l300k(layer=5), vs_dp4a=False)


def test_tc_causal_row_groups_with_ties():
    x = gen.causal64(L=20000, R=64)
    _check(x, rows=[0, 1, 2, 3, 4, 37, 62, 63])


def test_tc_causal_odd_row_count():
    x = gen.causal64(L=3001, R=7)      # groups of 4 and 3 rows
    _check(x)


def test_tc_varlen_batch():
    x = gen.make_inputs("v", seed=5, lengths=[0, 77, 128, 3000, 129, 20000], **gen.MLA,
                        key_mode="near_parallel")
    _check(x)


def test_tc_int8_extremes():
    x = gen.l64k(L=3000)
    rng = np.random.default_rng(1)
    x.k_idx[:] = rng.choice(np.array([-128, 127, -127, 0, 1], np.int8), x.k_idx.shape)
    x.q_idx[:] = rng.choice(np.array([-128, 127, -1], np.int8), x.q_idx.shape)
    x.w_idx[:] = rng.choice(np.array([1, 4], np.int32), x.w_idx.shape)
    _check(x)


def test_tc_without_relu_negative_weights():
    x = gen.l64k(L=5000)
    x.w_idx[:] = np.where(np.arange(64) % 3 == 0, -3, 2).astype(np.int32)[None]
    _check(x, relu=False)


@pytest.mark.parametrize("H_i,D_i", [(32, 64), (32, 128), (128, 128), (64, 64)])
def test_tc_head_and_dim_variants(H_i, D_i):
    x = gen.make_inputs("hd", seed=H_i * 7 + D_i, lengths=[2500, 900], rows_per_request=[3, 2],
                        row_len=[2500, 2400, 2000, 900, 700], H_i=H_i, D_i=D_i, H_q=16,
                        D_k=64, D_v=64, k=256, softmax_scale=0.125)
    _check(x)


def test_tc_biased_path_at_its_exactness_limit():
    # D_i * max|q| * 1279 < 2^24 allows a declared bound of 102 at D_i = 128:
    # values at +-102 keep every partial sum of the biased MMA exact in fp32.
    x = gen.l64k(L=2000)
    rng = np.random.default_rng(7)
    x.q_idx[:] = rng.choice(np.array([-102, 102, 101, -1], np.int8), x.q_idx.shape)
    x.k_idx[:] = rng.choice(np.array([-102, 102, 0], np.int8), x.k_idx.shape)
    x.w_idx[:] = 1
    _check_one(x, None, True, True, 102)


def test_tc_fp8_path_at_its_exactness_limit():
    # A declared bound of 11 at D_i = 128 selects e4m3 operands (every |v| <= 16 is
    # an e4m3 integer, and 128 * 11^2 < 2^14 keeps each head's dot small): values
    # at +-11 everywhere must still give bit-exact scores.
    x = gen.l64k(L=3000)
    rng = np.random.default_rng(11)
    x.q_idx[:] = rng.choice(np.array([-11, 11, 7, -3, 0], np.int8), x.q_idx.shape)
    x.k_idx[:] = rng.choice(np.array([-11, 11, -10, 9, 1], np.int8), x.k_idx.shape)
    _check_one(x, None, True, True, 11)
    _check_one(x, None, False, True, 11)


def _worst_case_rows(n, D_i=128, v=11):
    """Deterministic int8 rows at +-v that drive each head's dot product to its
    extremes: all +v, all -v, alternating signs (complete cancellation), signs
    per block of 32 (one MMA K-step of the e4m3 mode), half and half, zero."""
    d = np.arange(D_i)
    pats = [np.full(D_i, v), np.full(D_i, -v), np.where(d % 2 == 0, v, -v),
            np.where((d // 32) % 2 == 0, v, -v), np.where(d < D_i // 2, v, -v),
            np.zeros(D_i, np.int64), np.where((d // 32) % 2 == 0, -v, v)]
    return np.stack([pats[i % len(pats)] for i in range(n)]).astype(np.int8)


@pytest.mark.parametrize("rows", [1, 2])
def test_tc_fp8_worst_case_dots_at_the_bound(rows):
    # Declared bound 11: e4m3 operands.  Every key and query value is +-11 or 0,
    # so a head's dot reaches 128 * 11^2 = 15488 (and -15488 without ReLU), and
    # every partial sum over a K-step of 32 is at its largest magnitude (3872 per
    # step); with w = 4 on every head the score reaches 64 * 4 * 15488.
    x = gen.causal64(L=3000, R=rows) if rows > 1 else gen.l64k(L=3000)
    x.k_idx[:] = _worst_case_rows(x.k_idx.shape[0])
    rng = np.random.default_rng(12)
    for r in range(x.R):
        q = _worst_case_rows(64)
        x.q_idx[r] = q[rng.permutation(64)]
    x.q_idx[0, 0] = 11                     # head 0 of row 0 against all +11 keys: +15488
    x.w_idx[:] = 4
    ref = oracle.indexer_scores(x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len)
    assert ref[0].max() >= 4 * 15488
    _check_one(x, None, True, True, 11)
    _check_one(x, None, False, True, 11)


def test_tc_fp8_with_128_column_accumulators():
    # 32 heads x 4 rows per request fill 128 accumulator columns per tile in the
    # e4m3 mode; the two tile parities must still own separate accumulators.
    x = gen.make_inputs("f4", seed=21, lengths=[3000, 1500], rows_per_request=[4, 4],
                        row_len=[3000, 2990, 2500, 100, 1500, 1400, 1499, 7], H_i=32, D_i=128,
                        H_q=16, D_k=64, D_v=64, k=256, softmax_scale=0.125)
    qk = value_bound(x)
    assert qk <= 11
    _check_one(x, None, True, True, qk)


@pytest.mark.parametrize("H_i,R,L", [(128, 1, 307200), (32, 8, 150000)])
def test_tc_two_accumulators_many_tiles_per_cta(H_i, R, L):
    # 128 accumulator columns per tile (128 heads of one row, or 4 rows x 32
    # heads) leave room for two accumulators: each CTA here takes dozens of
    # tiles, so the MMA issuers cycle through both many times.
    x = gen.make_inputs("acc2", seed=H_i + R, lengths=[L], rows_per_request=[R],
                        row_len=[L - R + 1 + i for i in range(R)], H_i=H_i, D_i=128, H_q=16,
                        D_k=64, D_v=64, k=256, softmax_scale=0.125)
    for qk in (value_bound(x), 0):   # e4m3 operands, then exact fp16
        _check_one(x, None, True, False, qk)

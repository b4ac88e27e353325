"""Pins of the oracle's indexer front end (CPU only): hand-worked examples,
closed forms of the affine projection, invariants of the quantisation, and the
bound that ties the integer operands back to the real-valued indexer score.

The weight format is the 8-bit affine group quantisation that
"GLM-5.3-Flash-Alis-MLX-4bit" (page 3, the Recipe table and the note under it)
keeps the DSA indexer projections in: groups of 64 inputs, one scale and one
bias per group, codes 0..255.
"""
import numpy as np
import pytest

import dsa_inputs as gen
import oracle


def _bits(vals):
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    f = np.asarray(vals, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def _weights(codes, scales, biases):
    return (np.asarray(codes, dtype=np.uint8), _bits(scales), _bits(biases))


def test_dequantize_hand_worked_example():
    # Two outputs over d = 128 (two groups of 64).
    codes = np.zeros((2, 128), dtype=np.uint8)
    codes[0, 0], codes[0, 70] = 10, 3
    codes[1, :] = 255
    W = oracle.dequantize_affine(*_weights(codes, [[0.5, 2.0], [1 / 128, 1 / 64]], [[-1.0, 0.25], [-1.0, -2.0]]))
    assert W[0, 0] == 0.5 * 10 - 1.0 == 4.0
    assert W[0, 1] == -1.0                      # code 0 in group 0: the bias alone
    assert W[0, 70] == 2.0 * 3 + 0.25 == 6.25   # group 1 takes the second scale and bias
    assert W[0, 100] == 0.25
    assert np.all(W[1, :64] == 255 / 128 - 1.0) and np.all(W[1, 64:] == 255 / 64 - 2.0)
    # y = W x by hand for x = e_0 - 2 e_70 + 0.5 e_100, and the groups' other
    # inputs at zero: row 0: 4 - 12.5 + 0.125; row 1: 0.9921875 + 1.984375 * (-1.5).
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, 0], x[0, 70], x[0, 100] = 1.0, -2.0, 0.5
    xb = _bits(x)
    codes_q = np.zeros((2, 128), dtype=np.uint8)
    codes_q[:] = codes
    r = oracle.indexer_front_end(xb, _weights(codes_q, [[0.5, 2.0], [1 / 128, 1 / 64]],
                                              [[-1.0, 0.25], [-1.0, -2.0]]),
                                 _weights(np.zeros((1, 128)), [[1.0, 1.0]], [[0.0, 0.0]]),
                                 H_i=1, D_i=2, q_max=8, w_max=4)
    assert r["proj"][0, 0] == -8.375 and r["proj"][0, 1] == -1.984375


def test_front_end_hand_worked_quantisation():
    # x = e_0, so each projection is scale * code + bias of input 0:
    #   qf = [0.25 * 16 - 1, 0.25 * 0 - 1.25] = [3, -1.25]; wf = 0.5 * 4 = 2.
    # sigma = 3 / 8 = 0.375; q = [round(8), round(-3.33)] = [8, -3];
    # u = 2 * 0.375 = 0.75; tau = 0.75 / 4; w = round(4) = 4.
    x = np.zeros((1, 64), dtype=np.float32)
    x[0, 0] = 1.0
    cq = np.zeros((2, 64), dtype=np.uint8)
    cq[0, 0] = 16
    cw = np.zeros((1, 64), dtype=np.uint8)
    cw[0, 0] = 4
    r = oracle.indexer_front_end(_bits(x), _weights(cq, [[0.25], [0.25]], [[-1.0], [-1.25]]),
                                 _weights(cw, [[0.5]], [[0.0]]), H_i=1, D_i=2, q_max=8, w_max=4)
    assert r["proj"].tolist() == [[3.0, -1.25, 2.0]]
    assert r["q_idx"].tolist() == [[[8, -3]]]
    assert r["q_scale"].tolist() == [[0.375]]
    assert r["w_idx"].tolist() == [[4]]
    assert r["w_scale"].tolist() == [0.1875]


def test_one_hot_inputs_read_single_weights():
    # x = 2^e * e_i makes proj[o] = 2^e (scale[o, i // 64] * code[o, i] + bias[o, i // 64]),
    # computed here from the codes directly, not through dequantize_affine.
    f = gen.front_end(R=1, d=192, H_i=2, D_i=8, seed=7)
    cq, sq, bq = f.wq
    cw, sw, bw = f.ww
    for i, e in ((0, 0), (63, 3), (64, -2), (191, 1)):
        x = np.zeros((1, 192), dtype=np.float32)
        x[0, i] = 2.0 ** e
        r = oracle.indexer_front_end(_bits(x), f.wq, f.ww, 2, 8, q_max=127, w_max=4)
        g = i // 64
        want_q = (gen.bf16_bits_to_f64(sq[:, g]) * cq[:, i] + gen.bf16_bits_to_f64(bq[:, g])) * 2.0 ** e
        want_w = (gen.bf16_bits_to_f64(sw[:, g]) * cw[:, i] + gen.bf16_bits_to_f64(bw[:, g])) * 2.0 ** e
        np.testing.assert_array_equal(r["proj"][0, :16], want_q)
        np.testing.assert_array_equal(r["proj"][0, 16:], want_w)


def test_group_indicator_input_sums_codes():
    # x = 1 on the 64 inputs of group g: proj[o] = scale_g * sum(codes of the group) + 64 bias_g.
    f = gen.front_end(R=1, d=256, H_i=1, D_i=16, seed=3)
    cq, sq, bq = f.wq
    for g in range(4):
        x = np.zeros((1, 256), dtype=np.float32)
        x[0, 64 * g:64 * (g + 1)] = 1.0
        r = oracle.indexer_front_end(_bits(x), f.wq, f.ww, 1, 16, q_max=127, w_max=4)
        want = (gen.bf16_bits_to_f64(sq[:, g]) * cq[:, 64 * g:64 * (g + 1)].astype(np.int64).sum(axis=1)
                + 64 * gen.bf16_bits_to_f64(bq[:, g]))
        np.testing.assert_allclose(r["proj"][0, :16], want, rtol=1e-15, atol=0)


def test_quantisation_invariants():
    f = gen.front_end(R=3, d=320, H_i=4, D_i=32, seed=11)
    base = oracle.indexer_front_end(f.x, f.wq, f.ww, 4, 32, q_max=10, w_max=4)
    # Every head's largest |qf| maps to +-q_max; every code is within the bounds.
    qf = base["proj"][:, :128].reshape(3, 4, 32)
    am = np.abs(qf).argmax(axis=2)
    top = np.take_along_axis(base["q_idx"].astype(np.int64), am[:, :, None], axis=2)[:, :, 0]
    np.testing.assert_array_equal(np.abs(top), 10)
    assert np.abs(base["q_idx"]).max() <= 10 and np.abs(base["w_idx"]).max() == 4
    # Negated inputs: codes negate, scales stay (round half to even is odd-symmetric).
    neg = oracle.indexer_front_end(f.x ^ np.uint16(0x8000), f.wq, f.ww, 4, 32, q_max=10, w_max=4)
    np.testing.assert_array_equal(neg["q_idx"], -base["q_idx"])
    np.testing.assert_array_equal(neg["w_idx"], -base["w_idx"])
    np.testing.assert_array_equal(neg["q_scale"], base["q_scale"])
    np.testing.assert_array_equal(neg["w_scale"], base["w_scale"])
    # Doubled inputs (exact in bf16): codes unchanged, sigma doubles, tau x4.
    xd = gen.f32_to_bf16_bits((gen.bf16_bits_to_f64(f.x) * 2).astype(np.float32))
    dbl = oracle.indexer_front_end(xd, f.wq, f.ww, 4, 32, q_max=10, w_max=4)
    np.testing.assert_array_equal(dbl["q_idx"], base["q_idx"])
    np.testing.assert_array_equal(dbl["w_idx"], base["w_idx"])
    np.testing.assert_allclose(dbl["q_scale"], 2 * base["q_scale"], rtol=1e-14)
    np.testing.assert_allclose(dbl["w_scale"], 4 * base["w_scale"], rtol=1e-14)


def test_zero_input_gives_zero_codes_and_scales():
    f = gen.front_end(R=2, d=128, H_i=2, D_i=8, seed=5)
    r = oracle.indexer_front_end(np.zeros((2, 128), np.uint16), f.wq, f.ww, 2, 8, q_max=127, w_max=4)
    assert not r["q_idx"].any() and not r["w_idx"].any()
    assert not r["q_scale"].any() and not r["w_scale"].any()


@pytest.mark.parametrize("q_max,w_max", [(127, 16), (10, 4), (31, 1000)])
def test_integer_score_approximates_the_real_indexer_score(q_max, w_max):
    # With sigma_h = max|qf_h| / q_max and u_h = wf_h sigma_h, the real score
    # S = sum_h wf_h relu(qf_h . k) and tau * (integer score of q_idx, w_idx)
    # differ by at most sum_h (|wf_h| sigma_h / 2 + tau q_max / 2) * ||k||_1:
    # rounding moves each query element by <= sigma_h / 2 (relu is 1-Lipschitz)
    # and each head weight by <= tau / 2, times relu(q_h . k) <= q_max ||k||_1.
    H_i, D_i = 8, 32
    f = gen.front_end(R=2, d=384, H_i=H_i, D_i=D_i, seed=13)
    r = oracle.indexer_front_end(f.x, f.wq, f.ww, H_i, D_i, q_max=q_max, w_max=w_max)
    keys = gen.uniform_nibbles(99, 1, 50 * D_i).reshape(50, D_i).astype(np.int64)
    L = keys.shape[0]
    for row in range(2):
        qf = r["proj"][row, :H_i * D_i].reshape(H_i, D_i)
        wf = r["proj"][row, H_i * D_i:]
        S = (np.maximum(qf @ keys.T, 0) * wf[:, None]).sum(axis=0)
        ints = oracle.indexer_scores(r["q_idx"][row:row + 1], r["w_idx"][row:row + 1], keys.astype(np.int8),
                                     np.array([0, L]), np.array([0, 1]), np.array([L]))[0]
        A = r["w_scale"][row] * ints.astype(np.float64)
        bound = (np.abs(wf) * r["q_scale"][row] / 2 + r["w_scale"][row] * q_max / 2).sum() * np.abs(keys).sum(axis=1)
        assert np.all(np.abs(S - A) <= bound * (1 + 1e-12) + 1e-12)
        # and the bound is not vacuous: the approximation tracks the score
        assert np.corrcoef(S, A)[0, 1] > 0.9

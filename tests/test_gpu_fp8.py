"""Parity of the FP8-cache attention (DSA_FLAG_KV_FP8: E4M3 codes with one
fp32 scale per row, the FP8 KV storage of "glm53-tensorfold-spark", page 4)
with the CPU oracle, through the C ABI.

Bar as for the bf16 cache: scores and indices bit-exact (the cache format does
not touch selection); the bf16 output within max|d| <= 1e-2 and relative
L2 <= 5e-3 of the oracle's float64 attention over the dequantised rows."""
import numpy as np
import pytest

import dsa_inputs as gen
import oracle
from gpu_harness import assert_out_close, run_ops, run_step

pytestmark = pytest.mark.gpu


def _check(x, res, rows, check_lse=True):
    scores, idx, out = oracle.decode_step(x, rows=rows)
    req = x.row_request()
    for j, r in enumerate(rows):
        n = int(x.row_len[r])
        if "scores" in res:
            assert np.array_equal(res["scores"][r, :n], scores[j]), f"scores differ, row {r}"
        assert np.array_equal(res["idx"][r], idx[j]), f"indices differ, row {r}"
        assert res["nsel"][r] == min(x.k, n)
        assert_out_close(res["out"][r], out[j])
        if check_lse and res.get("lse") is not None and n > 0:
            lo, hi = int(x.offsets[req[r]]), int(x.offsets[req[r] + 1])
            sc = None if x.kv_scale is None else x.kv_scale[lo:hi]
            ref = oracle.attention_lse(x.q[r], x.kv[lo:hi], idx[j], x.softmax_scale, sc)
            np.testing.assert_allclose(res["lse"][r], ref, rtol=0, atol=2e-3)
    assert res["status"] == 0


def test_fp8_tiny_workload():
    x = gen.fp8_cache(gen.tiny())
    _check(x, run_ops(x), [0])


@pytest.mark.parametrize("L", [1000, 2049, 9000])
def test_fp8_mla_shapes(L):
    x = gen.fp8_cache(gen.l64k(L=L))
    _check(x, run_ops(x), [0])


def test_fp8_without_scales():
    x = gen.fp8_cache(gen.l64k(L=3000), with_scale=False)
    assert x.kv_scale is None
    _check(x, run_ops(x), [0])


def test_fp8_l64k_full_size():
    x = gen.fp8_cache(gen.l64k())
    _check(x, run_ops(x), [0])


def test_fp8_many_rows_loop_over_tiles():
    # 64 rows x 4 head groups: one cluster per (row, head group), so each CTA
    # takes 8 tiles and the staging buffer is refilled while a tile computes.
    x = gen.fp8_cache(gen.causal64(L=5000, R=64))
    _check(x, run_ops(x), [0, 31, 63])


def test_fp8_varlen_with_empty_and_short_requests():
    x = gen.fp8_cache(gen.make_inputs("varlen", seed=78, lengths=[0, 5, 300, 2048, 5000],
                                      **gen.MLA))
    res = run_ops(x)
    assert res["nsel"][0] == 0 and not res["out"][0].any()
    _check(x, res, [1, 2, 3, 4])


def test_fp8_decode_step_matches_ops_and_is_deterministic():
    # One decode row runs the single-row kernel; the three separate calls run
    # the clustered attention: the same selection, outputs each within the
    # tolerance of the oracle, and the step gives the same bits on every run.
    x = gen.fp8_cache(gen.l64k(L=20000))
    a = run_ops(x, lse=False)
    b = run_step(x)
    c = run_step(x)
    for key in ("idx", "nsel"):
        assert np.array_equal(a[key], b[key]), key
    for key in ("idx", "nsel", "out"):
        assert np.array_equal(b[key], c[key]), key
    _check(x, b, [0], check_lse=False)


@pytest.mark.parametrize("L", [1, 17, 2049, 9000])
def test_fp8_decode_step_single_row_kernel(L):
    x = gen.fp8_cache(gen.l64k(L=L))
    _check(x, run_step(x), [0], check_lse=False)


def test_fp8_decode_step_without_scales_and_with_subnormal_codes():
    x = gen.fp8_cache(gen.l64k(L=5000), with_scale=False)
    _check(x, run_step(x), [0], check_lse=False)
    y = gen.fp8_cache(gen.l64k(L=4000))
    rng = np.random.default_rng(22)
    mask = rng.random(y.kv.shape) < 0.05
    y.kv[mask] = rng.choice(np.r_[np.arange(8), np.arange(0x80, 0x88)].astype(np.uint8), int(mask.sum()))
    _check(y, run_step(y), [0], check_lse=False)


def test_fp8_decode_step_full_long_context_layer():
    x = gen.fp8_cache(gen.l300k(layer=2))
    _check(x, run_step(x), [0], check_lse=False)


def test_fp8_scales_are_applied():
    # Doubling every scale is not the same as the unscaled cache: the logits and
    # the values both double, and the output follows the oracle either way.
    x = gen.fp8_cache(gen.l64k(L=3000))
    y = gen.fp8_cache(gen.l64k(L=3000))
    y.kv_scale = (x.kv_scale * 2.0).astype(np.float32)
    rx, ry = run_ops(x), run_ops(y)
    assert not np.array_equal(rx["out"], ry["out"])
    _check(x, rx, [0])
    _check(y, ry, [0])


def test_fp8_zero_and_subnormal_codes():
    # Codes with a zero exponent field (zeros and subnormals) take the kernel's
    # other widening; plant them densely in every row.
    x = gen.fp8_cache(gen.l64k(L=4000))
    rng = np.random.default_rng(21)
    mask = rng.random(x.kv.shape) < 0.05
    x.kv[mask] = rng.choice(np.r_[np.arange(8), np.arange(0x80, 0x88)].astype(np.uint8), int(mask.sum()))
    _check(x, run_ops(x), [0])

"""A prefill chunk through the decode-step path: 2048 causal query rows of one
request at the end of a 10240-position context (the prefill step of 2,048
tokens of "GLM-5.3-Flash-Alis-MLX-4bit", page 3).  Every row selects its own
top-k among the positions it may see and attends over them.

Sampled rows are compared with the oracle (scores and indices bit-exact,
output within the tolerance); every row is checked for the properties that
define the ordered top-k of its (bit-exact on the samples) scores."""
import numpy as np
import pytest

import dsa_inputs as gen
import oracle
from gpu_harness import assert_out_close, run_ops, run_step, topk_properties

pytestmark = pytest.mark.gpu


def test_prefill_chunk_2048_rows():
    x = gen.prefill()
    res = run_ops(x)
    assert res["status"] == 0
    topk_properties(res["scores"], res["idx"], res["nsel"], x.row_len, x.k)
    rows = [0, 1, 777, 2047]
    scores, idx, out = oracle.decode_step(x, rows=rows)
    for j, r in enumerate(rows):
        n = int(x.row_len[r])
        assert np.array_equal(res["scores"][r, :n], scores[j]), f"scores differ, row {r}"
        assert np.array_equal(res["idx"][r], idx[j]), f"indices differ, row {r}"
        assert_out_close(res["out"][r], out[j])


def test_prefill_chunk_decode_step_equals_ops():
    x = gen.prefill(L=6144, R=1024)
    a = run_ops(x, lse=False)
    b = run_step(x)
    for key in ("idx", "nsel", "out"):
        assert np.array_equal(a[key], b[key]), key
    assert b["status"] == 0
    scores, idx, out = oracle.decode_step(x, rows=[5, 1023])
    for j, r in enumerate([5, 1023]):
        assert np.array_equal(b["idx"][r], idx[j])
        assert_out_close(b["out"][r], out[j])

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
from gpu_harness import assert_out_close, run_ops, run_step

pytestmark = pytest.mark.gpu


def _topk_properties(scores, idx, nsel, row_len, k):
    """For every row: nsel = min(k, len); the selection is distinct positions
    in range, ordered by (score desc, position asc), padded with -1; no
    unselected position scores above the last selected score T; and of the
    positions scoring exactly T, the lowest ones are the selected ones."""
    for r in range(idx.shape[0]):
        n = int(row_len[r])
        m = min(k, n)
        assert nsel[r] == m
        sel = idx[r, :m]
        assert (idx[r, m:] == -1).all()
        assert sel.min() >= 0 and sel.max() < n and np.unique(sel).size == m
        s = scores[r, :n].astype(np.int64)
        key = s[sel]
        assert (np.diff(key) <= 0).all(), f"row {r}: scores not descending"
        eq = np.diff(key) == 0
        assert (np.diff(sel)[eq] > 0).all(), f"row {r}: ties not by position"
        if m < n:
            T = key[-1]
            rest = np.ones(n, bool)
            rest[sel] = False
            assert s[rest].max() <= T, f"row {r}: an unselected score beats the threshold"
            tied_out = np.nonzero(rest & (s == T))[0]
            tied_in = sel[key == T]
            if tied_out.size:
                assert tied_in.max() < tied_out.min(), f"row {r}: ties at T not lowest positions"


def test_prefill_chunk_2048_rows():
    x = gen.prefill()
    res = run_ops(x)
    assert res["status"] == 0
    _topk_properties(res["scores"], res["idx"], res["nsel"], x.row_len, x.k)
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

"""Bounded device waits made to run out on purpose (include/dsa_testing.h),
without faulting or hanging the GPU: the top-k's grid barrier with one CTA
that never arrives, the attention's gather barrier armed for rows that are
never copied, and the indexer's key-tile barrier armed for a tile that is never
loaded.  Each call must return within milliseconds with DSA_DEVICE_TIMEOUT in
the status word; the attention must leave the rows it could not compute
untouched; and the same workspace and context must then give exact results."""
import time

import numpy as np
import pytest

import dsa_inputs as gen
import oracle
from gpu_harness import assert_out_close

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000   # 1 ms


def _topk_problem(dsa, rows):
    import torch
    R = len(rows)
    lens = np.array([len(r) for r in rows], np.int32)
    L_max = int(lens.max())
    scores = np.zeros((R, L_max), np.int32)
    for i, r in enumerate(rows):
        scores[i, :len(r)] = r
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    t = dict(offsets=torch.from_numpy(offsets).cuda(),
             row_offsets=torch.arange(R + 1, dtype=torch.int32, device="cuda"),
             row_len=torch.from_numpy(lens).cuda())
    prob = dsa.Problem(R=R, B=R, H_i=64, D_i=128, H_q=64, D_k=576, D_v=512, k=2048, L_max=L_max,
                       L_total=int(offsets[-1]), softmax_scale=1.0, **t)
    return prob, t, torch.from_numpy(scores).cuda()


@pytest.mark.parametrize("skip_cta", [0, 5])
def test_topk_grid_barrier_with_a_missing_arrival(skip_cta):
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    rng = np.random.default_rng(31)
    rows = [rng.integers(-10**6, 10**6, 300000).astype(np.int32)]
    prob, t, s = _topk_problem(dsa, rows)
    ws = dsa.alloc_workspace(prob)
    idx = torch.full((1, 2048), -9, dtype=torch.int32, device="cuda")
    nsel = torch.full((1,), -9, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dsa.dsa_test_topk_missing_arrival(prob, s, idx, nsel, ws, skip_cta, LIMIT_NS)
    bits = dsa.dsa_read_device_status(ws)
    assert time.perf_counter() - t0 < 5.0
    assert bits & dsa.DSA_DEVICE_TIMEOUT
    assert dsa.dsa_get_device_status(ws) == dsa.DSA_ERR_TIMEOUT
    # The context and the workspace still work.
    dsa.dsa_topk(prob, s, idx, nsel, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    assert np.array_equal(idx.cpu().numpy()[0].astype(np.int64), oracle.topk_indices(rows[0], 2048))


@pytest.mark.parametrize("make", [lambda: gen.tiny(L=3000), lambda: gen.l64k(L=9000)])
def test_attention_gather_that_never_lands_leaves_output_untouched(make):
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    x = make()
    prob, t = dsa.upload_inputs(x)
    ws = dsa.alloc_workspace(prob)
    ref_idx = oracle.topk_indices(oracle.indexer_scores(
        x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len)[0], x.k)
    idx = torch.from_numpy(ref_idx.astype(np.int32)[None]).cuda()
    nsel = torch.tensor([min(x.k, int(x.row_len[0]))], dtype=torch.int32, device="cuda")
    out = torch.full((1, x.H_q, x.D_v), 0x1234, dtype=torch.int16, device="cuda")
    lse = torch.full((1, x.H_q), 7.5, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dsa.dsa_test_attn_missing_gather(prob, idx, nsel, out, lse, ws, LIMIT_NS)
    bits = dsa.dsa_read_device_status(ws)
    assert time.perf_counter() - t0 < 5.0
    assert bits & dsa.DSA_DEVICE_TIMEOUT
    assert (out.cpu().numpy() == 0x1234).all(), "a row whose gather ran out was written"
    assert (lse.cpu().numpy() == 7.5).all()
    dsa.dsa_sparse_attn(prob, idx, nsel, out, lse, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    ref = oracle.sparse_attention(x.q[0], x.kv, ref_idx, x.D_v, x.softmax_scale)
    assert_out_close(out.cpu().numpy().view(np.uint16)[0], ref)


def test_indexer_key_tile_that_never_lands():
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    x = gen.l64k(L=40000)
    prob, t = dsa.upload_inputs(x, qk_abs_max=10)
    ws = dsa.alloc_workspace(prob)
    s = torch.full((1, x.L_max), -99, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dsa.dsa_test_indexer_missing_tile(prob, s, ws, LIMIT_NS)
    bits = dsa.dsa_read_device_status(ws)
    assert time.perf_counter() - t0 < 5.0
    assert bits & dsa.DSA_DEVICE_TIMEOUT
    dsa.dsa_index_scores(prob, s, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    ref = oracle.indexer_scores(x.q_idx, x.w_idx, x.k_idx, x.offsets, x.row_offsets, x.row_len)[0]
    assert np.array_equal(s.cpu().numpy()[0], ref)
    # A whole decode step on the same workspace afterwards.
    idx = torch.empty((1, x.k), dtype=torch.int32, device="cuda")
    out = torch.empty((1, x.H_q, x.D_v), dtype=torch.int16, device="cuda")
    dsa.dsa_decode_step(prob, idx, None, out, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    assert np.array_equal(idx.cpu().numpy()[0].astype(np.int64), oracle.topk_indices(ref, x.k))


def test_hooks_validate_their_arguments():
    import dsa_sparse_attention_03_gb300 as dsa
    x = gen.tiny(L=3000)
    prob, t = dsa.upload_inputs(x)
    ws = dsa.alloc_workspace(prob)
    import torch
    s = torch.zeros((1, x.L_max), dtype=torch.int32, device="cuda")
    with pytest.raises(dsa.DsaError):          # no tensor-memory operand at D_i = 32
        dsa.dsa_test_indexer_missing_tile(prob, s, ws, LIMIT_NS)
    with pytest.raises(dsa.DsaError):          # limit out of range
        dsa.dsa_test_indexer_missing_tile(prob, s, ws, 0)

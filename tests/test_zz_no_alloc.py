"""dsa_topk_static (the top-k with the library's fixed scratch instead of a
caller workspace) against the CPU oracle's full stable sort and against
dsa_topk, two calls in a row per problem after a call on other data has left
its own contents in the scratch; and its rejection of problems whose scratch
would not fit.  Collected last, so it also runs after every other GPU test in
the same process."""
import numpy as np
import pytest

import dsa_inputs as gen
import oracle

pytestmark = pytest.mark.gpu


def _scores(dsa, x, qk):
    import torch
    prob, t = dsa.upload_inputs(x, qk_abs_max=qk)
    ws = dsa.alloc_workspace(prob)
    s = torch.zeros((x.R, max(1, x.L_max)), dtype=torch.int32, device="cuda")
    dsa.dsa_index_scores(prob, s, ws)
    return prob, t, ws, s


def _prime(dsa):
    """A top-k on unrelated data (an all-equal row, the exact fallback), so the
    static scratch holds another problem's state before the calls under test."""
    import torch
    L = 9000
    t = dict(offsets=torch.tensor([0, L], dtype=torch.int32, device="cuda"),
             row_offsets=torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
             row_len=torch.tensor([L], dtype=torch.int32, device="cuda"))
    p = dsa.Problem(R=1, B=1, H_i=64, D_i=128, H_q=64, D_k=576, D_v=512, k=2048, L_max=L,
                    L_total=L, softmax_scale=1.0, **t)
    s = torch.full((1, L), 7, dtype=torch.int32, device="cuda")
    idx = torch.empty((1, 2048), dtype=torch.int32, device="cuda")
    dsa.dsa_topk_static(p, s, idx, None)
    torch.cuda.synchronize()
    assert idx.cpu().numpy()[0].tolist() == list(range(2048))


def _pair(dsa, prob, ws, s, R, k):
    import torch
    _prime(dsa)
    idx_w = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
    nsel_w = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_topk(prob, s, idx_w, nsel_w, ws)
    outs = []
    for _ in range(2):   # two calls in a row reuse the same static scratch
        idx_s = torch.full((R, k), -9, dtype=torch.int32, device="cuda")
        nsel_s = torch.full((R,), -9, dtype=torch.int32, device="cuda")
        dsa.dsa_topk_static(prob, s, idx_s, nsel_s)
        outs.append((idx_s.cpu().numpy(), nsel_s.cpu().numpy()))
    torch.cuda.synchronize()
    return (idx_w.cpu().numpy(), nsel_w.cpu().numpy()), outs


@pytest.mark.parametrize("make", [
    lambda: gen.tiny(),
    lambda: gen.l64k(layer=1),
    lambda: gen.causal64(L=20000, R=16),
    lambda: gen.make_inputs("v", seed=3, lengths=[0, 900, 5000, 70000], **gen.MLA,
                            key_mode="near_parallel"),
])
def test_static_scratch_matches_oracle_and_workspace_topk(make):
    import dsa_sparse_attention_03_gb300 as dsa
    x = make()
    prob, _, ws, s = _scores(dsa, x, 0)
    ref, outs = _pair(dsa, prob, ws, s, x.R, x.k)
    scores = s.cpu().numpy()
    for r in range(x.R):
        n = int(x.row_len[r])
        want = oracle.topk_indices(scores[r, :n], x.k)
        assert np.array_equal(ref[0][r], want), f"dsa_topk row {r}"
        assert ref[1][r] == min(x.k, n)
    for idx_s, nsel_s in outs:
        assert np.array_equal(idx_s, ref[0])
        assert np.array_equal(nsel_s, ref[1])


def test_static_scratch_rejects_problem_that_does_not_fit():
    import ctypes
    import dsa_sparse_attention_03_gb300 as dsa
    lib = dsa.lib()
    fake = 1 << 20   # host validation rejects the call before anything is enqueued
    p = dsa.Problem(R=512, B=512, H_i=64, D_i=128, H_q=64, D_k=576, D_v=512, k=2048,
                    L_max=4096, L_total=512 * 4096, softmax_scale=1 / 24)
    for f in ("offsets", "row_offsets", "row_len"):
        setattr(p.c, f, fake)
    st = lib.dsa_topk_static(ctypes.byref(p.c), fake, fake, fake, None)
    assert st == dsa.DSA_ERR_UNSUPPORTED
    msg = lib.dsa_last_error_string().decode()
    assert "static scratch" in msg and str(4 << 20) in msg

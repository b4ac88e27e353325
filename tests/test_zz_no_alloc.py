"""dsa_topk_static (the top-k with the library's fixed scratch instead of a
caller workspace) against dsa_topk, two calls in a row per problem; and its
rejection of problems whose scratch would not fit.  Collected last, so it also
runs after every other GPU test in the same process."""
import numpy as np
import pytest

import dsa_inputs as gen

pytestmark = pytest.mark.gpu


def _scores(dsa, x, qk):
    import torch
    prob, t = dsa.upload_inputs(x, qk_abs_max=qk)
    ws = dsa.alloc_workspace(prob)
    s = torch.zeros((x.R, max(1, x.L_max)), dtype=torch.int32, device="cuda")
    dsa.dsa_index_scores(prob, s, ws)
    return prob, t, ws, s


def _pair(dsa, prob, ws, s, R, k):
    import torch
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
def test_static_scratch_matches_workspace_topk(make):
    import dsa_sparse_attention_03_gb300 as dsa
    x = make()
    prob, _, ws, s = _scores(dsa, x, 0)
    ref, outs = _pair(dsa, prob, ws, s, x.R, x.k)
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

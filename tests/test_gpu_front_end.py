"""The indexer front end on the GPU against the oracle (dsa_indexer_front_end,
include/dsa_front_end.h).

The kernel projects in fp32, so the comparison is not bit-exact.  What is
checked, element by element:

* each projection within 2^-17 * T of the oracle's exact value, where T is the
  sum of the magnitudes of the terms that make it up,
  T[o] = sum_g (|scale_g| sum_{i in g} |code_i x_i| + |bias_g| sum_{i in g} |x_i|):
  the kernel's sums are a fixed tree of at most ~100 fp32 roundings deep
  (16-term lane dot, 5-level warp tree, item chain, the group's bias term), each
  costing at most 2^-24 of the running magnitude, and 2^-17 = 128 * 2^-24;
* each code within 1/2 + e of the oracle's exact ratio (qf / sigma or u / tau),
  with e the propagated bound of those projection errors through the quantiser
  (plus a few fp32 roundings): a code may differ from the exact-arithmetic code
  only where the exact ratio lies within e of a rounding midpoint;
* the scales within their propagated bounds;
* and almost all codes equal to the oracle's (boundary cases are rare).
"""
import numpy as np
import pytest

import dsa_inputs as gen
import oracle

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24
GAMMA = 2.0 ** -17


def _term_sums(f):
    """T[r, o]: sum of |terms| of every projection (host arithmetic for the bound)."""
    X = np.abs(gen.bf16_bits_to_f64(f.x))                     # [R, d]
    out = []
    for codes, sc, bi in (f.wq, f.ww):
        s = np.abs(gen.bf16_bits_to_f64(sc))                  # [O, G]
        b = np.abs(gen.bf16_bits_to_f64(bi))
        O, d = codes.shape
        cx = np.einsum("oi,ri->roi", codes.astype(np.float64), X).reshape(X.shape[0], O, d // 64, 64).sum(axis=3)
        xs = X.reshape(X.shape[0], d // 64, 64).sum(axis=2)   # [R, G]
        out.append((cx * s[None]).sum(axis=2) + xs @ b.T)
    return np.concatenate(out, axis=1)


def _run(f, q_max, w_max, with_proj=True, x=None, ws_fill=0x3C):
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    dev = torch.device("cuda", 0)
    x = f.x if x is None else x
    prob = dsa.Problem(R=f.R, B=1, H_i=f.H_i, D_i=f.D_i, H_q=1, D_k=16, D_v=16, k=1, L_max=1,
                       L_total=1, softmax_scale=1.0, qk_abs_max=q_max, w_abs_max=w_max)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    xt = t(x.view(np.int16))
    wq = [t(f.wq[0]), t(f.wq[1].view(np.int16)), t(f.wq[2].view(np.int16))]
    ww = [t(f.ww[0]), t(f.ww[1].view(np.int16)), t(f.ww[2].view(np.int16))]
    ws = torch.empty(dsa.dsa_front_end_workspace_size(prob, f.d), dtype=torch.uint8, device=dev)
    ws.fill_(ws_fill)   # the front end must not rely on a clean workspace
    q_idx = torch.full((f.R, f.H_i, f.D_i), 99, dtype=torch.int8, device=dev)
    w_idx = torch.full((f.R, f.H_i), -99, dtype=torch.int32, device=dev)
    q_scale = torch.full((f.R, f.H_i), float("nan"), device=dev)
    w_scale = torch.full((f.R,), float("nan"), device=dev)
    proj = torch.full((f.R, f.H_i * f.D_i + f.H_i), float("nan"), device=dev) if with_proj else None
    dsa.dsa_indexer_front_end(prob, f.d, xt, wq, ww, q_idx, w_idx, ws, q_scale=q_scale,
                              w_scale=w_scale, proj=proj)
    torch.cuda.synchronize()
    return dict(q_idx=q_idx.cpu().numpy(), w_idx=w_idx.cpu().numpy(), q_scale=q_scale.cpu().numpy(),
                w_scale=w_scale.cpu().numpy(), proj=None if proj is None else proj.cpu().numpy())


def _check(f, got, q_max, w_max, x=None):
    x = f.x if x is None else x
    ref = oracle.indexer_front_end(x, f.wq, f.ww, f.H_i, f.D_i, q_max, w_max)
    g2 = gen.FrontEndInputs(f.name, f.R, f.d, f.H_i, f.D_i, x, f.wq, f.ww)
    tol = GAMMA * _term_sums(g2) + 1e-30                      # [R, O]
    R, H, D = f.R, f.H_i, f.D_i
    Oq = H * D
    if got["proj"] is not None:
        err = np.abs(got["proj"].astype(np.float64) - ref["proj"])
        assert np.all(err <= tol), f"projection error {np.max(err / tol):.3g} x its bound"
    qf = ref["proj"][:, :Oq].reshape(R, H, D)
    wf = ref["proj"][:, Oq:]
    t_q = tol[:, :Oq].reshape(R, H, D)
    t_w = tol[:, Oq:]
    a = np.abs(qf).max(axis=2)                                # [R, H]
    t_a = t_q.max(axis=2)
    sig = ref["q_scale"]
    # sigma
    sig_err = t_a / q_max + 2 * U32 * sig
    assert np.all(np.abs(got["q_scale"] - sig) <= sig_err + 1e-30)
    # query codes
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(a[:, :, None] > 0, qf * q_max / np.where(a > 0, a, 1)[:, :, None], 0.0)
        e_r = np.where(a[:, :, None] > 0,
                       (q_max * t_q + np.abs(ratio) * t_a[:, :, None]) / np.maximum(a - t_a, 1e-300)[:, :, None]
                       + 4 * U32 * np.abs(ratio), 0.0)
    cq = got["q_idx"].astype(np.float64)
    assert np.all(np.abs(cq) <= q_max)
    lim = np.clip(ratio, -q_max, q_max)
    assert np.all(np.abs(cq - lim) <= 0.5 + e_r + 1e-12), "query code off by more than the bound allows"
    assert np.mean(cq == ref["q_idx"]) > 0.999
    # head weights
    u = wf * sig
    e_u = np.abs(wf) * sig_err + sig * t_w + 2 * U32 * np.abs(u)
    m = np.abs(u).max(axis=1)                                  # [R]
    e_m = e_u.max(axis=1)
    tau = ref["w_scale"]
    assert np.all(np.abs(got["w_scale"] - tau) <= e_m / w_max + 2 * U32 * tau + 1e-30)
    with np.errstate(divide="ignore", invalid="ignore"):
        rw = np.where(m[:, None] > 0, u * w_max / np.where(m > 0, m, 1)[:, None], 0.0)
        e_rw = np.where(m[:, None] > 0,
                        w_max * (e_u + np.abs(u) * e_m[:, None] / np.where(m > 0, m, 1)[:, None])
                        / np.maximum(m - e_m, 1e-300)[:, None] + 4 * U32 * np.abs(rw), 0.0)
    cw = got["w_idx"].astype(np.float64)
    assert np.all(np.abs(cw) <= w_max)
    assert np.all(np.abs(cw - np.clip(rw, -w_max, w_max)) <= 0.5 + e_rw + 1e-12), "head weight off"
    assert np.mean(cw == ref["w_idx"]) > 0.99
    return ref


@pytest.mark.parametrize("R,d,H_i,D_i,q_max,w_max", [
    (1, 6144, 64, 128, 10, 4),     # the decode shape: 64 heads x 128, declared bounds 10 and 4
    (3, 512, 4, 32, 127, 16),      # the smallest width: one 512-input item per row
    (5, 1536, 8, 64, 31, 1000),    # 5 rows: a pass of 4 and a pass of 1
    (9, 512, 2, 256, 127, 4),      # 9 rows: passes of 4, 4 and 1
    (2, 1024, 1, 32, 8, 4),        # 33 output rows: one per CTA
])
def test_front_end_matches_oracle(R, d, H_i, D_i, q_max, w_max):
    f = gen.front_end(R=R, d=d, H_i=H_i, D_i=D_i, seed=1000 + R * 7 + d)
    got = _run(f, q_max, w_max)
    _check(f, got, q_max, w_max)


def test_front_end_many_rows_and_no_projection_output():
    # 40 rows (ten passes of 4), and proj = NULL (the projections stay in the workspace).
    f = gen.front_end(R=40, d=1024, H_i=16, D_i=64, seed=77)
    got = _run(f, 127, 8, with_proj=False)
    _check(f, got, 127, 8)


def test_front_end_zero_rows_and_determinism():
    f = gen.front_end(R=4, d=1024, H_i=8, D_i=128, seed=5)
    x = f.x.copy()
    x[2] = 0                                    # a zero hidden vector: zero codes and scales
    a = _run(f, 10, 4, x=x)
    ref = _check(f, a, 10, 4, x=x)
    assert not a["q_idx"][2].any() and not a["w_idx"][2].any()
    assert not a["q_scale"][2].any() and a["w_scale"][2] == 0
    assert ref["w_scale"][2] == 0
    b = _run(f, 10, 4, x=x, ws_fill=0xC3)
    for k in ("q_idx", "w_idx", "q_scale", "w_scale", "proj"):
        np.testing.assert_array_equal(a[k], b[k])

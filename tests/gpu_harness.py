"""Shared helpers of the GPU tests: run libdsa through its C ABI on seeded
inputs and compare with the CPU oracle (test infrastructure)."""
import numpy as np

import dsa_inputs as gen

ATOL = 1e-2      # max |out - oracle| on the bf16 attention output
RTOL_L2 = 5e-3   # ||out - oracle||_2 / ||oracle||_2


def value_bound(x):
    """The caller's declared bound on |q_idx| and |k_idx| (from the data)."""
    return int(max(np.abs(x.q_idx.astype(np.int32)).max(initial=0),
                   np.abs(x.k_idx.astype(np.int32)).max(initial=0), 1))


def run_ops(x, indexer="auto", relu=True, lse=True, scores_fill=-7, qk="data"):
    """dsa_index_scores -> dsa_topk -> dsa_sparse_attn; returns host arrays.
    qk: declared |q|,|k| bound ("data" = the inputs' own maximum, 0 = int8 range)."""
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    qk = value_bound(x) if qk == "data" else qk
    prob, t = dsa.upload_inputs(x, indexer=indexer, relu=relu, qk_abs_max=qk)
    ws = dsa.alloc_workspace(prob)
    ws.fill_(0xAB)  # the library must not rely on a clean workspace
    dev = ws.device
    scores = torch.full((x.R, max(x.L_max, 1)), scores_fill, dtype=torch.int32, device=dev)
    idx = torch.full((x.R, x.k), -5, dtype=torch.int32, device=dev)
    nsel = torch.full((x.R,), -5, dtype=torch.int32, device=dev)
    out = torch.full((x.R, x.H_q, x.D_v), 0x7FC0, dtype=torch.int16, device=dev)
    lse_t = torch.full((x.R, x.H_q), float("nan"), dtype=torch.float32, device=dev) if lse else None
    dsa.dsa_index_scores(prob, scores, ws)
    dsa.dsa_topk(prob, scores, idx, nsel, ws)
    dsa.dsa_sparse_attn(prob, idx, nsel, out, lse_t, ws)
    status = dsa.dsa_read_device_status(ws)
    torch.cuda.synchronize()
    return dict(scores=scores.cpu().numpy(), idx=idx.cpu().numpy().astype(np.int64),
                nsel=nsel.cpu().numpy(), out=out.cpu().numpy().view(np.uint16),
                lse=None if lse_t is None else lse_t.cpu().numpy(), status=status)


def run_step(x, indexer="auto", qk="data"):
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    qk = value_bound(x) if qk == "data" else qk
    prob, t = dsa.upload_inputs(x, indexer=indexer, qk_abs_max=qk)
    ws = dsa.alloc_workspace(prob)
    ws.fill_(0x5A)
    idx = torch.full((x.R, x.k), -5, dtype=torch.int32, device=ws.device)
    nsel = torch.full((x.R,), -5, dtype=torch.int32, device=ws.device)
    out = torch.empty((x.R, x.H_q, x.D_v), dtype=torch.int16, device=ws.device)
    dsa.dsa_decode_step(prob, idx, nsel, out, ws)
    status = dsa.dsa_read_device_status(ws)
    return dict(idx=idx.cpu().numpy().astype(np.int64), nsel=nsel.cpu().numpy(),
                out=out.cpu().numpy().view(np.uint16), status=status)


def assert_out_close(got_bits, ref):
    got = gen.bf16_bits_to_f64(got_bits)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    if not np.any(ref):
        assert not np.any(got), "expected an all-zero output"
        return
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= ATOL and rel <= RTOL_L2, f"max|d|={err:.3e} relL2={rel:.3e}"


def topk_properties(scores, idx, nsel, row_len, k):
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
        if m == 0:
            continue
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

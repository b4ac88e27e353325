"""Plain definitions of the DSA decode step (test infrastructure only).

Every function takes host numpy arrays in the library's layouts:

``q_idx`` int8 [R, H_i, D_i]   indexer query of each row, one vector per head
``w_idx`` int32 [R, H_i]       indexer head weights of each row
``k_idx`` int8 [L_total, D_i]  indexer keys, one per cached position (all heads)
``q``     bf16 bits [R, H_q, D_k] attention queries
``kv``    bf16 bits [L_total, D_k] latent cache rows (key = all D_k columns,
                                value = the first D_v columns); for an FP8
                                cache, E4M3 codes uint8 [L_total, D_k] with
``kv_scale`` float32 [L_total] per-row scales (None = all 1)
``offsets`` [B+1]      cache rows of request b are offsets[b]..offsets[b+1]-1
``row_offsets`` [B+1]  query rows of request b are row_offsets[b]..row_offsets[b+1]-1
``row_len`` [R]        row r sees request-local positions 0..row_len[r]-1
"""
from __future__ import annotations

import numpy as np

INT32_MIN = -(1 << 31)
INT32_MAX = (1 << 31) - 1


def _row_request(row_offsets, R):
    req = np.empty(R, dtype=np.int64)
    for b in range(len(row_offsets) - 1):
        req[int(row_offsets[b]):int(row_offsets[b + 1])] = b
    return req


def _bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_to_f64(codes):
    """Decode FP8 E4M3 codes (uint8) to float64, from the format's definition
    (OCP 8-bit floating point, E4M3): bit 7 is the sign, bits 6..3 the exponent
    field E (bias 7), bits 2..0 the mantissa M.  E = 0 encodes the subnormal
    M/8 * 2**-6; otherwise the value is (1 + M/8) * 2**(E - 7), except that
    E = 15 with M = 7 is NaN (the format has no infinities; the largest finite
    value is 1.75 * 2**8 = 448).  The stored format of the FP8 KV cache of
    "glm53-tensorfold-spark" (page 4), which does not name the variant; E4M3 is
    the reading taken.
    """
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    neg = (b >> 7) & 1
    e = (b >> 3) & 15
    m = (b & 7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & ((b & 7) == 7), np.nan, mag)
    return np.where(neg == 1, -mag, mag)


def _kv_rows_f64(kv_req, sel, kv_scale_req):
    """Rows ``sel`` of a request's cache as float64: bf16 bits widened exactly,
    or E4M3 codes (uint8) decoded and multiplied by their row's scale."""
    rows = np.asarray(kv_req)[sel]
    if rows.dtype == np.uint8:
        vals = e4m3_to_f64(rows)
        if kv_scale_req is not None:
            vals = vals * np.asarray(kv_scale_req, dtype=np.float64)[sel][:, None]
        return vals
    return _bf16_to_f64(rows)


def indexer_scores(q_idx, w_idx, k_idx, offsets, row_offsets, row_len, relu=True, rows=None):
    """Lightning-indexer scores, one int64 vector per row.

    For row r of request b and visible position t < row_len[r]:

        s[r, t] = sum_h  w[r, h] * max(0, sum_d q[r, h, d] * k[offsets[b] + t, d])

    (without the ``max(0, .)`` when ``relu`` is False).  The position is scored
    against every indexer head of the current query and the head results are
    combined with the query's own weights ("ds4 glm53-m3ultra", page 1: the
    search over all cached positions; the ReLU-weighted head sum is the reading
    taken where the pages give no formula).  Validity comes from each row's own
    length, never from the packed layout ("GLM-5.3-Flash-Alis-MLX-4bit", page 3,
    the indexer padding fix).

    Raises ``OverflowError`` if any score does not fit int32, the type the
    library's scores are stored in.
    """
    R = q_idx.shape[0]
    req = _row_request(row_offsets, R)
    out = []
    for r in (range(R) if rows is None else rows):
        b = int(req[r])
        lo = int(offsets[b])
        n = int(row_len[r])
        keys = k_idx[lo:lo + n].astype(np.int64)              # [n, D_i]
        qr = q_idx[r].astype(np.int64)                         # [H_i, D_i]
        dots = keys @ qr.T                                     # [n, H_i]
        if relu:
            dots = np.maximum(dots, 0)
        s = dots @ w_idx[r].astype(np.int64)                   # [n]
        if s.size and (s.min() < INT32_MIN or s.max() > INT32_MAX):
            raise OverflowError("indexer score outside int32")
        out.append(s)
    return out


def topk_indices(scores, k):
    """Ordered top-k of one row's scores.

    Returns int64 [k]: the positions of the min(k, n) largest scores, ordered by
    score descending and, among equal scores, by position ascending; entries past
    min(k, n) are -1.  A full stable sort of all n positions -- the plain
    definition of "same positions selected, same order" ("ds4 glm53-m3ultra",
    page 1), with the tie rule "lower index first".  A row with n <= k selects
    every position.
    """
    s = np.asarray(scores, dtype=np.int64)
    n = s.shape[0]
    order = np.argsort(-s, kind="stable")   # stable: equal scores keep index order
    m = min(k, n)
    out = np.full(k, -1, dtype=np.int64)
    out[:m] = order[:m]
    return out


def sparse_attention(q_row, kv_req, idx, D_v, softmax_scale, kv_scale_req=None):
    """Attention of every head of one query row over the selected latent rows.

    ``q_row`` bf16 bits [H_q, D_k]; ``kv_req`` bf16 bits [L_b, D_k] (the
    request's own cache rows), or E4M3 codes uint8 [L_b, D_k] whose row j is
    worth ``kv_scale_req[j]`` times the decoded codes (None = 1); ``idx`` the
    selected request-local positions (entries < 0 are unused).  In float64,
    with kv the rows' values, for head h:

        z_j  = softmax_scale * sum_{d < D_k} q[h, d] * kv[idx_j, d]
        p_j  = exp(z_j - max z) / sum_j' exp(z_j' - max z)
        o[h, c] = sum_j p_j * kv[idx_j, c]          for c < D_v

    -- attention over only the selected positions ("ds4 glm53-m3ultra", page 1),
    with keys and values read from one shared latent row per position (the
    latent, absorbed-MLA cache of "glm53-tensorfold-spark", page 4; value = the
    first D_v columns).  Returns float64 [H_q, D_v]; with no selected position
    the output is all zeros.
    """
    sel = np.asarray(idx)
    sel = sel[sel >= 0]
    H_q, D_k = q_row.shape
    if sel.size == 0:
        return np.zeros((H_q, D_v), dtype=np.float64)
    Q = _bf16_to_f64(q_row)                                   # [H_q, D_k]
    K = _kv_rows_f64(kv_req, sel, kv_scale_req)               # [n, D_k]
    z = softmax_scale * (Q @ K.T)                             # [H_q, n]
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    p = e / e.sum(axis=1, keepdims=True)
    return p @ K[:, :D_v]                                     # [H_q, D_v]


def attention_lse(q_row, kv_req, idx, softmax_scale, kv_scale_req=None):
    """Natural-log log-sum-exp of the scaled logits of each head over the
    selected rows, log(sum_j exp(z_j)) with z as in ``sparse_attention``;
    -inf when nothing is selected.  Returns float64 [H_q]."""
    sel = np.asarray(idx)
    sel = sel[sel >= 0]
    if sel.size == 0:
        return np.full(q_row.shape[0], -np.inf)
    z = softmax_scale * (_bf16_to_f64(q_row) @ _kv_rows_f64(kv_req, sel, kv_scale_req).T)
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def decode_step(inp, relu=True, rows=None):
    """Scores -> ordered top-k -> sparse attention for the rows of ``inp``
    (a ``DecodeInputs``-like object).  Returns (scores list, idx int64 [R', k],
    out float64 [R', H_q, D_v]) for the requested rows (all rows by default)."""
    rows = list(range(inp.R)) if rows is None else list(rows)
    req = _row_request(inp.row_offsets, inp.R)
    scores = indexer_scores(inp.q_idx, inp.w_idx, inp.k_idx, inp.offsets, inp.row_offsets,
                            inp.row_len, relu=relu, rows=rows)
    idx = np.stack([topk_indices(s, inp.k) for s in scores]) if rows else np.zeros((0, inp.k), np.int64)
    kv_scale = getattr(inp, "kv_scale", None)
    outs = []
    for j, r in enumerate(rows):
        b = int(req[r])
        lo, hi = int(inp.offsets[b]), int(inp.offsets[b + 1])
        sc = None if kv_scale is None else kv_scale[lo:hi]
        outs.append(sparse_attention(inp.q[r], inp.kv[lo:hi], idx[j], inp.D_v, inp.softmax_scale, sc))
    out = np.stack(outs) if outs else np.zeros((0, inp.H_q, inp.D_v))
    return scores, idx, out


def dequantize_affine(codes, scale_bits, bias_bits, group=64):
    """Weights stored as 8-bit affine codes with one scale and one bias per
    group of ``group`` consecutive inputs, as float64.

    ``codes`` uint8 [O, d]; ``scale_bits``, ``bias_bits`` bf16 bits [O, d / group].
    Weight (o, i) is ``scale[o, i // group] * codes[o, i] + bias[o, i // group]``
    -- the affine group quantisation that "GLM-5.3-Flash-Alis-MLX-4bit" (page 3,
    the Recipe table and the note under it) keeps the DSA indexer projections in:
    8 bits, groups of 64, packed in the standard MLX affine form (codes 0..255,
    scales and biases in the model's 16-bit type).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.float64)
    O, d = c.shape
    s = _bf16_to_f64(scale_bits).reshape(O, d // group)
    b = _bf16_to_f64(bias_bits).reshape(O, d // group)
    return c * np.repeat(s, group, axis=1) + np.repeat(b, group, axis=1)


def _round_half_even(v):
    return np.rint(v)   # numpy rounds halves to even


def indexer_front_end(x, wq, ww, H_i, D_i, q_max, w_max):
    """Indexer query and head weights of each row from its hidden vector.

    ``x`` bf16 bits [R, d]; ``wq`` = (codes [H_i * D_i, d], scales, biases) and
    ``ww`` = (codes [H_i, d], scales, biases), both in the 8-bit affine form of
    ``dequantize_affine``.  In float64, for each row:

        qf[h, :] = Wq[h * D_i : (h + 1) * D_i] @ x     (the indexer query, per head)
        wf[h]    = Ww[h] @ x                            (the head weight)

    then the integer operands the indexer takes (int8 q_idx, int32 w_idx within
    the declared bounds q_max and w_max):

        sigma_h  = max_j |qf[h, j]| / q_max
        q_idx    = clip(round(qf[h, j] / sigma_h), -q_max, q_max)
        u_h      = wf[h] * sigma_h
        tau      = max_h |u_h| / w_max
        w_idx    = clip(round(u_h / tau), -w_max, w_max)

    with round-half-to-even, and zero codes where sigma_h or tau is 0.  Since
    sigma_h > 0, sum_h wf_h max(0, qf_h . k) = sum_h u_h max(0, (qf_h / sigma_h) . k),
    so tau * (the integer score of q_idx, w_idx) approximates the score of the
    real-valued projections: each head's query scale folds into its weight.
    The pages fix only the weight format (page 3); the projection from one hidden
    vector, the per-head symmetric query scale and the per-row weight scale are
    the readings taken.  Returns a dict of float64 ``proj`` [R, H_i * D_i + H_i]
    (qf then wf), int8 ``q_idx`` [R, H_i, D_i], int32 ``w_idx`` [R, H_i], float64
    ``q_scale`` [R, H_i] (sigma) and ``w_scale`` [R] (tau).
    """
    X = _bf16_to_f64(x)
    R = X.shape[0]
    Wq = dequantize_affine(*wq)
    Ww = dequantize_affine(*ww)
    qf = (X @ Wq.T).reshape(R, H_i, D_i)
    wf = X @ Ww.T                                                  # [R, H_i]
    amax = np.abs(qf).max(axis=2)                                  # [R, H_i]
    sigma = amax / q_max
    safe = np.where(sigma > 0, sigma, 1.0)
    q = np.where(sigma[:, :, None] > 0, _round_half_even(qf / safe[:, :, None]), 0.0)
    q = np.clip(q, -q_max, q_max)
    u = wf * sigma
    tau = np.abs(u).max(axis=1) / w_max                            # [R]
    safe_t = np.where(tau > 0, tau, 1.0)
    w = np.where(tau[:, None] > 0, _round_half_even(u / safe_t[:, None]), 0.0)
    w = np.clip(w, -w_max, w_max)
    return {
        "proj": np.concatenate([qf.reshape(R, H_i * D_i), wf], axis=1),
        "q_idx": q.astype(np.int8),
        "w_idx": w.astype(np.int32),
        "q_scale": sigma,
        "w_scale": tau,
    }

"""dsa_topk on crafted score rows, against the oracle's full stable sort:
long random rows, the largest scores on a regular stride, a crowded threshold
bin and heavy ties (the exact fallback), scores spanning the whole int32 range
(rows of only INT32_MIN or only INT32_MAX included), and rows of every kind in
one call, with one row (survivors ranked across the grid) and with many rows
(each row's survivors sorted by one CTA; a row in the exact fallback resolved
by a pair of CTAs).  Scores are given directly, so each
path is reached on purpose."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

K = 2048


def _topk(rows, k=K, standalone=True):
    """rows: list of int32 arrays (one query row per request).  Runs dsa_topk
    (twice on the same workspace, to check that no state leaks between calls)
    and returns (idx [R, k], nsel [R])."""
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    R = len(rows)
    L_max = max(1, max(len(r) for r in rows))
    lens = np.array([len(r) for r in rows], dtype=np.int32)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    dev = "cuda"
    scores = np.full((R, L_max), -123, dtype=np.int32)
    for i, r in enumerate(rows):
        scores[i, :len(r)] = r
    t = dict(offsets=torch.from_numpy(offsets).to(dev),
             row_offsets=torch.arange(R + 1, dtype=torch.int32, device=dev),
             row_len=torch.from_numpy(lens).to(dev))
    prob = dsa.Problem(R=R, B=R, H_i=64, D_i=128, H_q=64, D_k=576, D_v=512, k=k, L_max=L_max,
                       L_total=int(offsets[-1]), softmax_scale=1.0, **t)
    ws = dsa.alloc_workspace(prob)
    ws.fill_(0xCD)
    s_dev = torch.from_numpy(scores).to(dev)
    outs = []
    for _ in range(2):
        idx = torch.full((R, k), -9, dtype=torch.int32, device=dev)
        nsel = torch.full((R,), -9, dtype=torch.int32, device=dev)
        dsa.dsa_topk(prob, s_dev, idx, nsel, ws)
        assert dsa.dsa_read_device_status(ws) == 0
        outs.append((idx.cpu().numpy().astype(np.int64), nsel.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    return outs[0]


def _check(rows, k=K):
    idx, nsel = _topk(rows, k)
    for i, r in enumerate(rows):
        ref = oracle.topk_indices(r, k)
        assert nsel[i] == min(k, len(r))
        assert np.array_equal(idx[i], ref), f"row {i}"


def test_random_long_row():
    rng = np.random.default_rng(3)
    _check([rng.integers(-10**6, 10**6, 300000, dtype=np.int64).astype(np.int32)])


def test_top_scores_on_a_regular_stride():
    # Every 37th position carries one of the largest scores (all distinct).
    L = 300000
    stride = -(-L // 8192)
    rng = np.random.default_rng(4)
    s = rng.integers(0, 1000, L).astype(np.int32)
    s[::stride] = 10**6 + np.arange(len(s[::stride]), dtype=np.int32)
    _check([s])


def test_twenty_thousand_scores_crowd_the_threshold():
    # 20000 positions share ten values just above the rest, so the threshold
    # bin holds thousands of positions (the exact fallback).
    L = 300000
    stride = -(-L // 8192)
    rng = np.random.default_rng(5)
    s = rng.integers(0, 1000, L).astype(np.int32)
    hot = np.arange(L)
    hot = hot[hot % stride != 0][:20000]
    s[hot] = 5000 + rng.integers(0, 10, len(hot))
    _check([s])


def test_all_equal_long_row_exact_path():
    _check([np.full(100000, 42, dtype=np.int32)])


def test_rows_of_every_kind_in_one_call():
    rng = np.random.default_rng(6)
    L = 150000
    stride = -(-L // 8192)
    hit = rng.integers(0, 50, L).astype(np.int32)
    hit[::stride] = 10**5
    rows = [rng.integers(-5000, 5000, L).astype(np.int32),   # random
            hit,                                            # heavy ties at the top, on a stride
            np.array([], dtype=np.int32),                   # empty
            rng.integers(0, 3, 1500).astype(np.int32),      # shorter than k
            rng.integers(-7, 7, 6000).astype(np.int32),     # few values: ties at T
            np.full(9000, -1, dtype=np.int32)]              # ties beyond the survivor cap
    _check(rows)


def test_small_k_and_lengths_around_8192():
    rng = np.random.default_rng(7)
    rows = [rng.integers(-100, 100, n).astype(np.int32) for n in (8191, 8192, 8193, 20000)]
    _check(rows, k=300)


def test_many_tied_rows_resolved_by_cta_pairs():
    # Ten or more rows, each in the exact fallback (the threshold bin holds more
    # than the survivor cap), so each is resolved by a pair of CTAs that split
    # the row at a tie block: lengths that split unevenly, rows whose winners
    # all lie in the second half, rows whose last tie taken lies in the first,
    # and a row with keys above the ties in both halves.
    rng = np.random.default_rng(12)
    rows = [rng.integers(0, 2, n).astype(np.int32) for n in (9000, 20001, 65537, 131071, 8193, 77777)]
    late = np.zeros(90000, np.int32)
    late[-10000:] = rng.integers(1, 3, 10000)          # ties at 2 only in the last 10000 positions
    early = np.zeros(90000, np.int32)
    early[:10000] = rng.integers(1, 3, 10000)          # ... only in the first 10000
    both = rng.integers(0, 2, 100000).astype(np.int32)
    both[[3, 60000, 99999]] = 7                        # a few keys above the ties, one in each half
    rows += [late, early, both, np.full(12345, 5, np.int32)]
    _check(rows)


def _int32_extreme_rows(rng):
    lo, hi = np.iinfo(np.int32).min, np.iinfo(np.int32).max
    full = rng.integers(lo, hi, 300000, dtype=np.int64, endpoint=True).astype(np.int32)
    full[[5, 77, 299999]] = hi
    full[[6, 1000, 250000]] = lo
    two = rng.choice(np.array([lo, hi], np.int32), 40000)
    few_max = np.full(30000, lo, np.int32)
    few_max[rng.choice(30000, 100, replace=False)] = hi
    near_edges = rng.choice(np.array([lo, lo + 1, -1, 0, 1, hi - 1, hi], np.int32), 50000)
    return [full, np.full(5000, lo, np.int32), np.full(5000, hi, np.int32), two, few_max,
            near_edges, np.array([hi, lo, 0], np.int32)]


def test_int32_extremes_one_row_at_a_time():
    # One row per call: the range and bins span INT32_MIN..INT32_MAX (the widest
    # bin shift), and the survivors are ranked across the grid.
    for row in _int32_extreme_rows(np.random.default_rng(8)):
        _check([row])


def test_int32_extremes_many_rows():
    # Eight or more rows in one call: each row's survivors are sorted by a CTA.
    rows = _int32_extreme_rows(np.random.default_rng(9))
    _check(rows + rows[:2])

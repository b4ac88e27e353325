"""dsa_check_bounds: the device check of the declared operand bounds (include/dsa.h).

The declared bounds qk_abs_max and w_abs_max are a promise the indexer relies
on (its exact operand format and the int32 overflow check).  The check reads
the operands and raises DSA_DEVICE_RANGE when one exceeds its bound."""
import numpy as np
import pytest

import dsa_inputs as gen

pytestmark = pytest.mark.gpu


def _bits(x, qk, wm, key_row0=0, key_rows=None):
    import torch
    import dsa_sparse_attention_03_gb300 as dsa
    prob, t = dsa.upload_inputs(x, qk_abs_max=qk, w_abs_max=wm)
    ws = torch.full((256,), 0x77, dtype=torch.uint8, device="cuda")   # status word cleared by the call
    dsa.dsa_check_bounds(prob, ws, key_row0=key_row0, key_rows=key_rows)
    return dsa.dsa_read_device_status(ws)


def test_data_within_its_own_bounds_is_clean():
    import dsa_sparse_attention_03_gb300 as dsa
    x = gen.l64k(L=20000)
    qk = int(max(np.abs(x.q_idx.astype(np.int32)).max(), np.abs(x.k_idx.astype(np.int32)).max()))
    assert _bits(x, qk, 4) == 0
    assert _bits(x, 0, 0) == 0             # 0 = the int8 range and w <= 4
    # one below the keys' largest magnitude: flagged
    assert _bits(x, qk - 1, 4) & dsa.DSA_DEVICE_RANGE


def test_a_single_key_byte_and_int8_min():
    import dsa_sparse_attention_03_gb300 as dsa
    x = gen.l64k(L=5000)
    x.k_idx = x.k_idx.copy()
    x.k_idx[4321, 77] = 11
    assert _bits(x, 10, 4) & dsa.DSA_DEVICE_RANGE
    assert _bits(x, 11, 4) == 0
    # rows 0..4320 only: the planted key is outside the checked range
    assert _bits(x, 10, 4, key_row0=0, key_rows=4321) == 0
    assert _bits(x, 10, 4, key_row0=4321, key_rows=1) & dsa.DSA_DEVICE_RANGE
    x.k_idx[4321, 77] = -128                # |-128| = 128 exceeds 127, and fits the unchecked 128
    assert _bits(x, 127, 4) & dsa.DSA_DEVICE_RANGE
    assert _bits(x, 128, 4) == 0


def test_query_and_weight_bounds():
    import dsa_sparse_attention_03_gb300 as dsa
    x = gen.l64k(L=3000)
    qk = int(max(np.abs(x.q_idx.astype(np.int32)).max(), np.abs(x.k_idx.astype(np.int32)).max()))
    assert _bits(x, qk, 3) & dsa.DSA_DEVICE_RANGE          # w in [1, 4]
    x.q_idx = x.q_idx.copy()
    x.q_idx[0, 63, 127] = qk + 1
    assert _bits(x, qk, 4) & dsa.DSA_DEVICE_RANGE
    assert _bits(x, qk + 1, 4) == 0
    x.w_idx = x.w_idx.copy()
    x.w_idx[0, 5] = -5                                       # |w| counts, not w
    assert _bits(x, qk + 1, 4) & dsa.DSA_DEVICE_RANGE
    assert _bits(x, qk + 1, 5) == 0

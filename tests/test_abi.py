"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, and validates arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__
    __graft_entry__.build()
    import dsa_sparse_attention_03_gb300 as m
    return m


def _declared():
    inc = os.path.join(ROOT, "include")
    txt = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    return sorted(set(re.findall(r"DSA_API\s+[\w\s\*]+?\b(dsa_\w+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(dsa):
    names = _declared()
    assert len(names) >= 8
    lib = ctypes.CDLL(dsa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(dsa.EXPORTS) == names


def test_struct_layout_matches_header(dsa):
    assert ctypes.sizeof(dsa.dsa_problem) == 136
    assert dsa.dsa_problem.L_total.offset == 40
    assert dsa.dsa_problem.q_idx.offset == 64
    assert dsa.dsa_problem.kv_scale.offset == 128   # appended after the ABI-100 fields
    assert dsa.dsa_version() == 101


def _prob(dsa, **kw):
    base = dict(R=1, B=1, H_i=64, D_i=128, H_q=64, D_k=576, D_v=512, k=2048, L_max=65536,
                L_total=65536, softmax_scale=1 / 24)
    base.update(kw)
    return dsa.Problem(**base)


def test_workspace_size_grows_with_rows_and_length(dsa):
    a = dsa.dsa_workspace_size(_prob(dsa))
    b = dsa.dsa_workspace_size(_prob(dsa, L_max=307200, L_total=307200))
    c = dsa.dsa_workspace_size(_prob(dsa, R=2, B=2))
    d = dsa.dsa_workspace_size(_prob(dsa, R=32, B=32))
    assert 0 < a < b and c < d
    assert a % 256 == 0
    # One query row (the single-row step) reserves the attention units'
    # partials: 128 units x 64 heads x 512 fp16 values at k = 2048.
    assert a > 128 * 64 * 512 * 2
    assert dsa.dsa_decode_step_kernels(_prob(dsa)) == 2
    assert dsa.dsa_decode_step_kernels(_prob(dsa, R=2, B=2)) == 3


def test_host_validation_rejects_before_launch(dsa):
    lib = dsa.lib()
    fake = 1 << 20
    # A misaligned workspace: even if a shape check under test failed to fire,
    # the workspace check would still reject the call before any launch.
    ws = ctypes.c_void_p(fake + 16)

    def status(null=False, **kw):
        p = _prob(dsa, **kw)
        if not null:
            for f in ("q_idx", "w_idx", "k_idx", "q", "kv", "offsets", "row_offsets", "row_len"):
                setattr(p.c, f, fake)
        return lib.dsa_decode_step(ctypes.byref(p.c), fake, None, fake, ws, 1 << 40, None)

    assert status(null=True) == dsa.DSA_ERR_INVALID_ARG            # null pointers
    assert status(D_i=48) == dsa.DSA_ERR_UNSUPPORTED
    assert status(k=0) == dsa.DSA_ERR_UNSUPPORTED
    assert status(k=5000) == dsa.DSA_ERR_UNSUPPORTED
    assert status(D_v=600) == dsa.DSA_ERR_UNSUPPORTED
    assert status(H_q=200) == dsa.DSA_ERR_UNSUPPORTED
    assert status(B=0) == dsa.DSA_ERR_UNSUPPORTED
    assert status(w_abs_max=1 << 20) == dsa.DSA_ERR_OVERFLOW_RISK
    assert b"2^31" in lib.dsa_last_error_string()
    assert lib.dsa_workspace_size(ctypes.byref(_prob(dsa, R=-1).c)) == 0
    assert b"R=-1" in lib.dsa_last_error_string()
    assert status(flags=0x400) == dsa.DSA_ERR_INVALID_ARG          # unknown flag bit
    assert b"flag" in lib.dsa_last_error_string()
    p = _prob(dsa, flags=dsa.DSA_FLAG_KV_FP8)
    for f in ("q_idx", "w_idx", "k_idx", "q", "kv", "offsets", "row_offsets", "row_len"):
        setattr(p.c, f, fake)
    p.c.kv_scale = fake + 2                                         # misaligned scales
    assert lib.dsa_sparse_attn(ctypes.byref(p.c), fake, None, fake, None, ws, 1 << 40,
                               None) == dsa.DSA_ERR_INVALID_ARG
    assert b"kv_scale" in lib.dsa_last_error_string()


def test_misaligned_and_small_workspace_rejected(dsa):
    lib = dsa.lib()
    p = dsa.Problem(R=1, B=1, H_i=4, D_i=32, H_q=8, D_k=64, D_v=64, k=256, L_max=4096,
                    L_total=4096, softmax_scale=1.0)
    fake = 1 << 20  # host validation only: nothing is launched when it fails
    for f in ("q_idx", "w_idx", "k_idx", "q", "kv", "offsets", "row_offsets", "row_len"):
        setattr(p.c, f, fake)
    need = dsa.dsa_workspace_size(p)
    st = lib.dsa_decode_step(ctypes.byref(p.c), fake, fake, fake, ctypes.c_void_p(fake + 16), need, None)
    assert st == dsa.DSA_ERR_INVALID_ARG and b"256-byte" in lib.dsa_last_error_string()
    st = lib.dsa_decode_step(ctypes.byref(p.c), fake, fake, fake, ctypes.c_void_p(fake), need - 1, None)
    assert st == dsa.DSA_ERR_INVALID_ARG and b"required" in lib.dsa_last_error_string()
    p.c.k_idx = fake + 4
    st = lib.dsa_index_scores(ctypes.byref(p.c), fake, ctypes.c_void_p(fake + 16), need, None)
    assert st == dsa.DSA_ERR_INVALID_ARG and b"k_idx" in lib.dsa_last_error_string()


def test_many_rows_reserve_no_cross_cluster_partials(dsa):
    # With many rows the attention runs one cluster per (row, head group), so
    # the workspace holds no cross-cluster partials: a 2048-row prefill chunk
    # needs its scores (R x L_max x 4), survivor keys (R x 4096 x 8) and
    # histograms, about 168 MB, not the 2.4 GB that 8 clusters' partials
    # would add.
    R, L = 2048, 10240
    n = dsa.dsa_workspace_size(_prob(dsa, R=R, B=1, L_max=L, L_total=L))
    assert R * L * 4 + R * 4096 * 8 < n < 200_000_000
    # one decode row keeps them (8 clusters of 4 CTAs per head group)
    one = dsa.dsa_workspace_size(_prob(dsa, R=1, B=1, L_max=L, L_total=L))
    assert one > 4 * 8 * 16 * 512 * 4


def test_binding_marshals_fp8_cache_and_flags(dsa):
    # Argument marshalling only (CPU tensors, nothing launched): an FP8 cache
    # sets DSA_FLAG_KV_FP8 and passes the codes and the row scales.
    import dsa_inputs as gen
    x = gen.fp8_cache(gen.tiny(L=300))
    prob, t = dsa.upload_inputs(x, device="cpu", indexer="dp4a", relu=False)
    c = prob.c
    assert c.flags == dsa.DSA_INDEXER_DP4A | dsa.DSA_FLAG_NO_RELU | dsa.DSA_FLAG_KV_FP8
    assert c.kv == t["kv"].data_ptr() and t["kv"].dtype.itemsize == 1 and tuple(t["kv"].shape) == (300, 64)
    assert c.kv_scale == t["kv_scale"].data_ptr() and t["kv_scale"].numel() == 300
    assert (c.R, c.B, c.L_max, c.L_total, c.D_k, c.D_v, c.k) == (1, 1, 300, 300, 64, 64, 256)
    y = gen.tiny(L=300)
    prob2, t2 = dsa.upload_inputs(y, device="cpu")
    assert prob2.c.flags == dsa.DSA_INDEXER_AUTO and not prob2.c.kv_scale
    assert t2["kv"].dtype.itemsize == 2


def test_front_end_validation_and_workspace(dsa):
    lib = dsa.lib()
    fake = 1 << 20   # host validation only: nothing is launched when it fails
    p = _prob(dsa, R=2, qk_abs_max=10, w_abs_max=4)
    n = dsa.dsa_front_end_workspace_size(p, 6144)
    O = 64 * 128 + 64
    assert n % 256 == 0 and n >= 2 * (O + 3) // 4 * 4 * 4 + 2 * 64 * 4 + 256
    assert lib.dsa_front_end_workspace_size(ctypes.byref(p.c), 640) == 0   # not a multiple of 512
    assert b"multiple of 512" in lib.dsa_last_error_string()
    w = dsa.dsa_affine_weights(fake, fake, fake)
    ws = ctypes.c_void_p(fake)

    def call(prob=p, d=6144, x=fake, wq=w, ww=w, q=fake, wi=fake, ws=ws, nbytes=n):
        return lib.dsa_indexer_front_end(ctypes.byref(prob.c), d, x, ctypes.byref(wq), ctypes.byref(ww),
                                         q, wi, None, None, None, ws, nbytes, None)

    assert call(x=None) == dsa.DSA_ERR_INVALID_ARG
    assert call(x=fake + 8) == dsa.DSA_ERR_INVALID_ARG and b"16-byte" in lib.dsa_last_error_string()
    assert call(wq=dsa.dsa_affine_weights(fake + 4, fake, fake)) == dsa.DSA_ERR_INVALID_ARG
    assert call(wq=dsa.dsa_affine_weights(fake, fake + 2, fake)) == dsa.DSA_ERR_INVALID_ARG
    assert call(ww=dsa.dsa_affine_weights(fake, None, fake)) == dsa.DSA_ERR_INVALID_ARG
    assert call(nbytes=n - 1) == dsa.DSA_ERR_INVALID_ARG and b"required" in lib.dsa_last_error_string()
    assert call(ws=ctypes.c_void_p(fake + 16)) == dsa.DSA_ERR_INVALID_ARG
    assert call(prob=_prob(dsa, R=2, D_i=48)) == dsa.DSA_ERR_UNSUPPORTED
    assert call(prob=_prob(dsa, R=2, qk_abs_max=200)) == dsa.DSA_ERR_INVALID_ARG
    assert call(d=65536) == dsa.DSA_ERR_UNSUPPORTED
    assert call(prob=_prob(dsa, R=0)) == dsa.DSA_OK    # nothing to do, nothing enqueued


def test_check_bounds_validation(dsa):
    lib = dsa.lib()
    fake = 1 << 20   # host validation only: nothing is launched when it fails
    p = _prob(dsa, R=1, qk_abs_max=10, w_abs_max=4, L_total=1000, L_max=1000)
    for f in ("q_idx", "w_idx", "k_idx"):
        setattr(p.c, f, fake)
    call = lambda r0, n, ws=fake, nb=256: lib.dsa_check_bounds(ctypes.byref(p.c), r0, n, ctypes.c_void_p(ws), nb, None)
    assert call(0, 1001) == dsa.DSA_ERR_INVALID_ARG and b"L_total" in lib.dsa_last_error_string()
    assert call(-1, 10) == dsa.DSA_ERR_INVALID_ARG
    assert call(0, 10, ws=fake + 16) == dsa.DSA_ERR_INVALID_ARG
    assert call(0, 10, nb=255) == dsa.DSA_ERR_INVALID_ARG
    p.c.k_idx = fake + 8
    assert call(0, 10) == dsa.DSA_ERR_INVALID_ARG and b"aligned" in lib.dsa_last_error_string()

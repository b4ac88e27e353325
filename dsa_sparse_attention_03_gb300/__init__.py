"""Python binding of libdsa (the DSA decode step for GB300, sm_103a).

Argument marshalling only: every step of the path runs in libdsa's CUDA
kernels, reached through its C ABI (``include/dsa.h``) with ctypes.  PyTorch
supplies device memory and streams.  There is no fallback: if the shared library
is missing this module raises at import.

Entry points mirror the C names::

    prob = Problem.from_tensors(...)          # sizes + device pointers
    ws = alloc_workspace(prob)                # caller-owned scratch
    dsa_index_scores(prob, scores, ws)
    dsa_topk(prob, scores, idx, nsel, ws)
    dsa_sparse_attn(prob, idx, nsel, out, lse, ws)
    dsa_decode_step(prob, idx, nsel, out, ws)
    dsa_read_device_status(ws)

and the indexer front end (``include/dsa_front_end.h``)::

    dsa_indexer_front_end(prob, d, x, wq, ww, q_idx, w_idx, ws_front, ...)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libdsa.so")

DSA_OK = 0
DSA_ERR_INVALID_ARG = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_OVERFLOW_RISK = 3
DSA_ERR_CUDA = 4
DSA_ERR_TIMEOUT = 5
DSA_ERR_DEVICE_INDEX = 6
DSA_ERR_RANGE = 7

DSA_DEVICE_TIMEOUT = 0x1
DSA_DEVICE_BAD_INDEX = 0x2
DSA_DEVICE_CAPACITY = 0x4
DSA_DEVICE_RANGE = 0x8

DSA_INDEXER_AUTO = 0
DSA_INDEXER_DP4A = 1
DSA_INDEXER_TC = 2
DSA_FLAG_NO_RELU = 0x100
DSA_FLAG_KV_FP8 = 0x200

INDEXERS = {"auto": DSA_INDEXER_AUTO, "dp4a": DSA_INDEXER_DP4A, "tc": DSA_INDEXER_TC}

# Symbols the header declares (checked by the ABI test).
EXPORTS = ("dsa_version", "dsa_last_error_string", "dsa_indexer_kind", "dsa_decode_step_kernels",
           "dsa_workspace_size",
           "dsa_index_scores",
           "dsa_topk", "dsa_topk_static", "dsa_sparse_attn", "dsa_decode_step",
           "dsa_read_device_status", "dsa_get_device_status", "dsa_check_bounds",
           # include/dsa_front_end.h
           "dsa_front_end_workspace_size", "dsa_indexer_front_end",
           # include/dsa_testing.h
           "dsa_test_topk_missing_arrival", "dsa_test_attn_missing_gather",
           "dsa_test_indexer_missing_tile")


class dsa_problem(ctypes.Structure):
    _fields_ = [
        ("R", ctypes.c_int32), ("B", ctypes.c_int32), ("H_i", ctypes.c_int32),
        ("D_i", ctypes.c_int32), ("H_q", ctypes.c_int32), ("D_k", ctypes.c_int32),
        ("D_v", ctypes.c_int32), ("k", ctypes.c_int32), ("L_max", ctypes.c_int32),
        ("flags", ctypes.c_int32), ("L_total", ctypes.c_int64),
        ("qk_abs_max", ctypes.c_int32), ("w_abs_max", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float), ("reserved0", ctypes.c_int32),
        ("q_idx", ctypes.c_void_p), ("w_idx", ctypes.c_void_p), ("k_idx", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("kv", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
        ("row_offsets", ctypes.c_void_p), ("row_len", ctypes.c_void_p),
        ("kv_scale", ctypes.c_void_p),
    ]


class dsa_affine_weights(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


class DsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libdsa status {status}: {message}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libdsa is not built ({LIB_PATH} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(dsa_problem)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.dsa_version.restype = ctypes.c_int
    lib.dsa_last_error_string.restype = ctypes.c_char_p
    lib.dsa_indexer_kind.restype = ctypes.c_int
    lib.dsa_indexer_kind.argtypes = [P]
    lib.dsa_decode_step_kernels.restype = ctypes.c_int
    lib.dsa_decode_step_kernels.argtypes = [P]
    lib.dsa_workspace_size.restype = sz
    lib.dsa_workspace_size.argtypes = [P]
    lib.dsa_front_end_workspace_size.restype = sz
    lib.dsa_front_end_workspace_size.argtypes = [P, ctypes.c_int32]
    W = ctypes.POINTER(dsa_affine_weights)
    for name, args in (
        ("dsa_index_scores", [P, vp, vp, sz, vp]),
        ("dsa_topk", [P, vp, vp, vp, vp, sz, vp]),
        ("dsa_topk_static", [P, vp, vp, vp, vp]),
        ("dsa_sparse_attn", [P, vp, vp, vp, vp, vp, sz, vp]),
        ("dsa_decode_step", [P, vp, vp, vp, vp, sz, vp]),
        ("dsa_read_device_status", [vp, vp, ctypes.POINTER(ctypes.c_int32)]),
        ("dsa_get_device_status", [vp, vp]),
        ("dsa_check_bounds", [P, ctypes.c_int64, ctypes.c_int64, vp, sz, vp]),
        ("dsa_indexer_front_end", [P, ctypes.c_int32, vp, W, W, vp, vp, vp, vp, vp, vp, sz, vp]),
        ("dsa_test_topk_missing_arrival", [P, vp, vp, vp, vp, sz, ctypes.c_int, ctypes.c_int64, vp]),
        ("dsa_test_attn_missing_gather", [P, vp, vp, vp, vp, vp, sz, ctypes.c_int64, vp]),
        ("dsa_test_indexer_missing_tile", [P, vp, vp, sz, ctypes.c_int64, vp]),
    ):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = args
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def _check(status: int) -> None:
    if status != DSA_OK:
        raise DsaError(status, _lib.dsa_last_error_string().decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Problem:
    """Sizes plus device tensors of one decode-step problem (see include/dsa.h).

    The tensors are kept referenced for the lifetime of the object.  ``L_max``
    and ``L_total`` are host values; ``from_tensors`` computes them from
    ``row_len``/``offsets`` (a device read) unless given.
    """

    def __init__(self, **kw):
        self._keep = {}
        s = dsa_problem()
        for f, _ in dsa_problem._fields_:
            v = kw.get(f)
            if v is None:
                continue
            if hasattr(v, "data_ptr"):
                self._keep[f] = v
                setattr(s, f, v.data_ptr())
            else:
                setattr(s, f, v)
        self.c = s

    @classmethod
    def from_tensors(cls, *, q_idx, w_idx, k_idx, q, kv, offsets, row_offsets, row_len, k,
                     softmax_scale, D_v=0, L_max=None, L_total=None, indexer="auto", relu=True,
                     qk_abs_max=0, w_abs_max=0, kv_fp8=False, kv_scale=None):
        R = int(row_len.shape[0])
        B = int(offsets.shape[0]) - 1
        if L_max is None:
            L_max = int(row_len.max().item()) if R else 0
        if L_total is None:
            L_total = int(offsets[-1].item())
        flags = (INDEXERS[indexer] | (0 if relu else DSA_FLAG_NO_RELU)
                 | (DSA_FLAG_KV_FP8 if kv_fp8 else 0))
        H_i, D_i = (int(q_idx.shape[1]), int(q_idx.shape[2])) if q_idx is not None else (0, 0)
        H_q, D_k = (int(q.shape[1]), int(q.shape[2])) if q is not None else (0, 0)
        return cls(R=R, B=B, H_i=H_i, D_i=D_i, H_q=H_q, D_k=D_k, D_v=int(D_v), k=int(k),
                   L_max=int(L_max), flags=flags, L_total=int(L_total), qk_abs_max=qk_abs_max,
                   w_abs_max=w_abs_max, softmax_scale=float(softmax_scale), q_idx=q_idx,
                   w_idx=w_idx, k_idx=k_idx, q=q, kv=kv, offsets=offsets,
                   row_offsets=row_offsets, row_len=row_len, kv_scale=kv_scale)

    def set(self, **kw):
        for f, v in kw.items():
            if hasattr(v, "data_ptr"):
                self._keep[f] = v
                v = v.data_ptr()
            setattr(self.c, f, v)
        return self

    def __getattr__(self, name):
        if name in ("c", "_keep"):
            raise AttributeError(name)
        return getattr(self.c, name)


def upload_inputs(inp, device="cuda", indexer="auto", relu=True, qk_abs_max=0, w_abs_max=0):
    """Copy a host problem (numpy arrays named as in include/dsa.h: q_idx,
    w_idx, k_idx, q, kv, offsets, row_offsets, row_len, plus k, D_v,
    softmax_scale; an FP8 cache has ``kv_format == "e4m3"``, kv as uint8 codes
    and ``kv_scale`` float32 or None) to ``device``.  Returns (Problem, dict of
    device tensors)."""
    import numpy as np
    import torch

    def dev(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)

    fp8 = getattr(inp, "kv_format", "bf16") == "e4m3"
    t = dict(
        q_idx=dev(inp.q_idx, torch.int8), w_idx=dev(inp.w_idx, torch.int32),
        k_idx=dev(inp.k_idx, torch.int8),
        q=dev(np.asarray(inp.q).view(np.int16), torch.int16),
        kv=(dev(np.asarray(inp.kv, dtype=np.uint8), torch.uint8) if fp8
            else dev(np.asarray(inp.kv).view(np.int16), torch.int16)),
        offsets=dev(inp.offsets, torch.int32), row_offsets=dev(inp.row_offsets, torch.int32),
        row_len=dev(inp.row_len, torch.int32))
    sc = getattr(inp, "kv_scale", None) if fp8 else None
    t["kv_scale"] = None if sc is None else dev(np.asarray(sc, dtype=np.float32), torch.float32)
    L_max = int(np.max(inp.row_len)) if len(inp.row_len) else 0
    prob = Problem.from_tensors(k=inp.k, D_v=inp.D_v, softmax_scale=inp.softmax_scale,
                                L_max=L_max, L_total=int(inp.offsets[-1]), indexer=indexer,
                                relu=relu, qk_abs_max=qk_abs_max, w_abs_max=w_abs_max,
                                kv_fp8=fp8, **t)
    return prob, t


def dsa_decode_step_kernels(prob: Problem) -> int:
    """Kernels one dsa_decode_step launches for this problem (2 or 3)."""
    return _lib.dsa_decode_step_kernels(ctypes.byref(prob.c))


def dsa_indexer_kind(prob: Problem) -> int:
    return _lib.dsa_indexer_kind(ctypes.byref(prob.c))


def indexer_kind(prob: Problem) -> str:
    return {DSA_INDEXER_DP4A: "dp4a", DSA_INDEXER_TC: "tc"}.get(dsa_indexer_kind(prob), "invalid")


def dsa_version() -> int:
    return _lib.dsa_version()


def dsa_workspace_size(prob: Problem) -> int:
    n = _lib.dsa_workspace_size(ctypes.byref(prob.c))
    if n == 0:
        raise DsaError(DSA_ERR_INVALID_ARG, _lib.dsa_last_error_string().decode())
    return n


def alloc_workspace(prob: Problem, device="cuda"):
    import torch
    return torch.empty(dsa_workspace_size(prob), dtype=torch.uint8, device=device)


def dsa_index_scores(prob: Problem, scores, ws, stream=None) -> None:
    _check(_lib.dsa_index_scores(ctypes.byref(prob.c), _ptr(scores), _ptr(ws), ws.numel(),
                                 _stream(stream)))


def dsa_topk(prob: Problem, scores, idx, nsel, ws, stream=None) -> None:
    _check(_lib.dsa_topk(ctypes.byref(prob.c), _ptr(scores), _ptr(idx), _ptr(nsel), _ptr(ws),
                         ws.numel(), _stream(stream)))


def dsa_topk_static(prob: Problem, scores, idx, nsel, stream=None) -> None:
    """dsa_topk with the library's fixed 4 MiB scratch instead of a workspace
    (see include/dsa.h: calls must not overlap)."""
    _check(_lib.dsa_topk_static(ctypes.byref(prob.c), _ptr(scores), _ptr(idx), _ptr(nsel),
                                _stream(stream)))


def dsa_sparse_attn(prob: Problem, idx, nsel, out, lse, ws, stream=None) -> None:
    _check(_lib.dsa_sparse_attn(ctypes.byref(prob.c), _ptr(idx), _ptr(nsel), _ptr(out),
                                _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))


def dsa_decode_step(prob: Problem, idx, nsel, out, ws, stream=None) -> None:
    _check(_lib.dsa_decode_step(ctypes.byref(prob.c), _ptr(idx), _ptr(nsel), _ptr(out),
                                _ptr(ws), ws.numel(), _stream(stream)))


# Test hooks (include/dsa_testing.h): one bounded device wait made to run out.

def dsa_test_topk_missing_arrival(prob: Problem, scores, idx, nsel, ws, skip_cta, limit_ns,
                                  stream=None) -> None:
    _check(_lib.dsa_test_topk_missing_arrival(ctypes.byref(prob.c), _ptr(scores), _ptr(idx),
                                              _ptr(nsel), _ptr(ws), ws.numel(), int(skip_cta),
                                              int(limit_ns), _stream(stream)))


def dsa_test_attn_missing_gather(prob: Problem, idx, nsel, out, lse, ws, limit_ns,
                                 stream=None) -> None:
    _check(_lib.dsa_test_attn_missing_gather(ctypes.byref(prob.c), _ptr(idx), _ptr(nsel),
                                             _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                             int(limit_ns), _stream(stream)))


def dsa_test_indexer_missing_tile(prob: Problem, scores, ws, limit_ns, stream=None) -> None:
    _check(_lib.dsa_test_indexer_missing_tile(ctypes.byref(prob.c), _ptr(scores), _ptr(ws),
                                              ws.numel(), int(limit_ns), _stream(stream)))


def dsa_check_bounds(prob: Problem, ws, key_row0=0, key_rows=None, stream=None) -> None:
    """Device check of the declared bounds (include/dsa.h); read the result
    with dsa_read_device_status."""
    n = int(prob.c.L_total) - int(key_row0) if key_rows is None else int(key_rows)
    _check(_lib.dsa_check_bounds(ctypes.byref(prob.c), int(key_row0), n, _ptr(ws), ws.numel(),
                                 _stream(stream)))


def dsa_get_device_status(ws, stream=None) -> int:
    """Synchronises the stream; returns DSA_OK, DSA_ERR_TIMEOUT or
    DSA_ERR_DEVICE_INDEX from the device status word (raises on other errors)."""
    st = _lib.dsa_get_device_status(_ptr(ws), _stream(stream))
    if st not in (DSA_OK, DSA_ERR_TIMEOUT, DSA_ERR_DEVICE_INDEX, DSA_ERR_RANGE):
        _check(st)
    return st


def dsa_read_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns the device status bits (raises on
    TIMEOUT / BAD_INDEX with the bits in ``DsaError.status``)."""
    bits = ctypes.c_int32(0)
    st = _lib.dsa_read_device_status(_ptr(ws), _stream(stream), ctypes.byref(bits))
    if st not in (DSA_OK, DSA_ERR_TIMEOUT, DSA_ERR_DEVICE_INDEX, DSA_ERR_RANGE):
        _check(st)
    return bits.value


# Indexer front end (include/dsa_front_end.h).

def affine_weights(codes, scales, biases) -> dsa_affine_weights:
    """The three device tensors of one 8-bit affine weight matrix."""
    return dsa_affine_weights(codes.data_ptr(), scales.data_ptr(), biases.data_ptr())


def dsa_front_end_workspace_size(prob: Problem, d: int) -> int:
    n = _lib.dsa_front_end_workspace_size(ctypes.byref(prob.c), int(d))
    if n == 0:
        raise DsaError(DSA_ERR_INVALID_ARG, _lib.dsa_last_error_string().decode())
    return n


def dsa_indexer_front_end(prob: Problem, d: int, x, wq, ww, q_idx, w_idx, ws, q_scale=None,
                          w_scale=None, proj=None, stream=None) -> None:
    """``wq``/``ww``: (codes, scales, biases) device tensors or dsa_affine_weights."""
    if not isinstance(wq, dsa_affine_weights):
        wq = affine_weights(*wq)
    if not isinstance(ww, dsa_affine_weights):
        ww = affine_weights(*ww)
    _check(_lib.dsa_indexer_front_end(ctypes.byref(prob.c), int(d), _ptr(x), ctypes.byref(wq),
                                      ctypes.byref(ww), _ptr(q_idx), _ptr(w_idx), _ptr(q_scale),
                                      _ptr(w_scale), _ptr(proj), _ptr(ws), ws.numel(),
                                      _stream(stream)))

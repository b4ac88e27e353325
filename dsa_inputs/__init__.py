"""Seeded synthetic inputs for the DSA decode step.

This module only draws random numbers and lays them out in the shapes of the
workloads; it holds none of the method's arithmetic (no scoring, selection or
attention).  Both the CPU oracle and the CUDA path are fed from here, and only
from here.

Random source: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-style: draw ``i``
of a stream is ``mix64(state0 + (i + 1) * GOLDEN_GAMMA)`` with the finaliser
``mix64`` of that paper, so any element can be produced independently of the
others and large tensors are generated in parallel chunks.  Each tensor has its
own stream, ``state0 = mix64(seed ^ (tag * GOLDEN_GAMMA))``.

Derived distributions (all defined on 64-bit draws ``u``):

* ``U{-8..7}`` int8 (the only uniform integer range of the workloads): the 16
  nibbles of one draw, value ``nibble - 8`` -- exactly uniform.
* ``U{lo..hi}`` for other ranges: ``lo + ((u >> 32) * n) >> 32`` with
  ``n = hi - lo + 1`` (Lemire's multiply-shift; bias below ``n / 2**32``).
* Bernoulli(p): ``(u >> 11) * 2**-53 < p``.
* N(0, 1): Box-Muller on the two 32-bit halves of one draw,
  ``r = sqrt(-2 ln(((u >> 32) + 1) / 2**32))``, ``theta = 2 pi (u & 0xffffffff) / 2**32``,
  giving ``r cos(theta)`` and ``r sin(theta)`` for two consecutive elements.
* bf16: the normal (times a scale) is rounded to float32, then to bf16 with
  round-to-nearest-even on the float32 bit pattern; stored as uint16 bits.

Workloads (the DSA decode step of a GLM-5.3-Flash-style layer, as described on
"ds4 glm53-m3ultra" (page 1: selection over ~2048 positions at 62k and 300k
context) and "GLM-5.3-Flash-Alis-MLX-4bit" (page 3: the per-row validity of the
indexer)):

* ``tiny``      : 1 query, L=4096, indexer 4 heads x 32, top-k 256, 8 attention
                  heads over a shared K=V latent of width 64; queries N(0,1)/8.
* ``l64k``      : 1 query, L=65536, indexer 64 x 128 with 10% of the keys
                  near-parallel to the query, top-k 2048, 64 heads over a
                  576-wide latent (512 value columns + 64 rope), scale 1/24.
* ``l300k``     : as ``l64k`` at L=307200, one independent layer per ``layer``.
* ``batch32``   : 32 requests, lengths U[4096, 131072], packed caches.
* ``causal64``  : 64 causal query rows over L=131072 whose indexer keys come
                  from only 16 distinct vectors (heavy ties at the threshold).
* ``prefill``   : a 2048-row causal prefill chunk at the end of a 10240-position
                  context ("GLM-5.3-Flash-Alis-MLX-4bit", page 3: a prefill
                  step of 2,048 tokens, and the gathered sparse prefill over
                  query chunks), keys as ``l64k``.

``front_end(...)`` draws the inputs of the indexer front end: one hidden vector
per query row, x ~ N(0, 1) in bf16, and synthetic 8-bit affine weights for the
query projection [H_i * D_i, d] and the head-weight projection [H_i, d]
("GLM-5.3-Flash-Alis-MLX-4bit", page 3: the indexer projections at 8 bits in
groups of 64, MLX affine form).  Codes are U{0..255}; each group of 64 inputs
has scale s0 * U{192..320} / 256 and bias -scale * U{120..135}, both rounded to
bf16, with s0 = sqrt(12) / (255 sqrt(d)), so each weight has standard deviation
about 1 / sqrt(d) and each projection is about N(0, 1).  No trained weights
exist here; these stand in for them.

``fp8_cache(x)`` turns any of them into the same problem over an FP8 latent
cache ("glm53-tensorfold-spark", page 4: FP8 KV storage), stored the way a cache
writer would store it: per row j, scale_j = max_d |kv[j, d]| / 448 (float32;
1 for an all-zero row) and code[j, d] = e4m3(kv[j, d] / scale_j), rounded to
nearest even by PyTorch's float8_e4m3fn cast.  The decode step consumes the
codes and scales as given; this writer is not part of it.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

GOLDEN_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

# Stream tags, one per tensor kind.
TAG_Q_IDX = 1
TAG_W_IDX = 2
TAG_K_IDX = 3
TAG_NEAR_PICK = 4
TAG_NEAR_NOISE = 5
TAG_Q = 6
TAG_KV = 7
TAG_LENGTHS = 8
TAG_DISTINCT_VEC = 9
TAG_DISTINCT_PICK = 10
TAG_FE_X = 11
TAG_FE_CODES = 12      # + 0 (query projection) or + 3 (head-weight projection)
TAG_FE_SCALE = 13
TAG_FE_BIAS = 14

_CHUNK = 1 << 22


def mix64(z: int) -> int:
    """SplitMix64 finaliser on a Python int (used for per-stream seeds)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def stream_seed(seed: int, tag: int) -> int:
    return mix64((seed ^ ((tag * GOLDEN_GAMMA) & _MASK64)) & _MASK64)


def _draws_chunk(state0: int, start: int, n: int) -> np.ndarray:
    z = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    z *= np.uint64(GOLDEN_GAMMA)
    z += np.uint64(state0)
    z ^= z >> np.uint64(30)
    z *= np.uint64(_M1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_M2)
    z ^= z >> np.uint64(31)
    return z


def _parallel(fn, n: int, out: np.ndarray, per_draw: int) -> np.ndarray:
    """Fill ``out`` (flat) from draws [0, n) in chunks; ``fn(draws) -> values``."""
    starts = list(range(0, n, _CHUNK))

    def work(s):
        m = min(_CHUNK, n - s)
        out[s * per_draw:(s + m) * per_draw] = fn(s, m)

    if len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    return out


def draws(seed: int, tag: int, n: int, start: int = 0) -> np.ndarray:
    """``n`` raw 64-bit draws of stream (seed, tag), beginning at counter ``start``."""
    st = stream_seed(seed, tag)
    out = np.empty(n, dtype=np.uint64)
    return _parallel(lambda s, m: _draws_chunk(st, start + s, m), n, out, 1)


def uniform_nibbles(seed: int, tag: int, n: int) -> np.ndarray:
    """``n`` int8 values U{-8..7}: sixteen 4-bit fields per draw, low nibble first."""
    st = stream_seed(seed, tag)
    nd = (n + 15) // 16
    out = np.empty(nd * 16, dtype=np.int8)

    def fn(s, m):
        u = _draws_chunk(st, s, m)
        shifts = (np.arange(16, dtype=np.uint64) * np.uint64(4))[None, :]
        nib = (u[:, None] >> shifts) & np.uint64(15)
        return (nib.astype(np.int16) - 8).astype(np.int8).reshape(-1)

    _parallel(fn, nd, out, 16)
    return out[:n]


def uniform_int(seed: int, tag: int, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` int64 values U{lo..hi} (multiply-shift on the high 32 bits)."""
    span = np.uint64(hi - lo + 1)
    u = draws(seed, tag, n)
    return ((u >> np.uint64(32)) * span >> np.uint64(32)).astype(np.int64) + lo


def bernoulli(seed: int, tag: int, n: int, p: float) -> np.ndarray:
    u = draws(seed, tag, n)
    return (u >> np.uint64(11)).astype(np.float64) * 2.0 ** -53 < p


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def normal_bf16(seed: int, tag: int, n: int, scale: float = 1.0) -> np.ndarray:
    """``n`` bf16 (uint16 bits) values of ``scale * N(0,1)`` via Box-Muller."""
    st = stream_seed(seed, tag)
    nd = (n + 1) // 2
    out = np.empty(nd * 2, dtype=np.uint16)

    def fn(s, m):
        u = _draws_chunk(st, s, m)
        u1 = ((u >> np.uint64(32)).astype(np.float64) + 1.0) * 2.0 ** -32
        u2 = (u & np.uint64(0xFFFFFFFF)).astype(np.float64) * 2.0 ** -32
        r = np.sqrt(-2.0 * np.log(u1))
        th = (2.0 * np.pi) * u2
        z = np.empty((m, 2), dtype=np.float64)
        z[:, 0] = r * np.cos(th)
        z[:, 1] = r * np.sin(th)
        if scale != 1.0:
            z *= scale
        return f32_to_bf16_bits(z.astype(np.float32).reshape(-1))

    _parallel(fn, nd, out, 2)
    return out[:n]


@dataclasses.dataclass
class DecodeInputs:
    """One DSA decode-step problem, host arrays only.

    Shapes: ``q_idx`` int8 [R, H_i, D_i]; ``w_idx`` int32 [R, H_i];
    ``k_idx`` int8 [L_total, D_i]; ``q`` bf16 bits [R, H_q, D_k];
    ``kv`` bf16 bits [L_total, D_k]; ``offsets`` int32 [B+1] (request b owns
    cache rows offsets[b]..offsets[b+1]-1); ``row_offsets`` int32 [B+1] (query
    rows of request b); ``row_len`` int32 [R] (positions row r may see).
    """
    name: str
    R: int
    B: int
    H_i: int
    D_i: int
    H_q: int
    D_k: int
    D_v: int
    k: int
    softmax_scale: float
    q_idx: np.ndarray
    w_idx: np.ndarray
    k_idx: np.ndarray
    q: np.ndarray
    kv: np.ndarray
    offsets: np.ndarray
    row_offsets: np.ndarray
    row_len: np.ndarray
    # "bf16": kv holds bf16 bits.  "e4m3": kv holds FP8 E4M3 codes (uint8) and
    # kv_scale float32 [L_total] the per-row scales (None = all 1).
    kv_format: str = "bf16"
    kv_scale: Optional[np.ndarray] = None

    @property
    def L_total(self) -> int:
        return int(self.offsets[-1])

    @property
    def L_max(self) -> int:
        return int(self.row_len.max()) if self.R else 0

    def row_request(self) -> np.ndarray:
        req = np.empty(self.R, dtype=np.int64)
        for b in range(self.B):
            req[self.row_offsets[b]:self.row_offsets[b + 1]] = b
        return req


def config_seed(cfg: int, layer: int = 0) -> int:
    return 0x0D5A0000 + 256 * cfg + layer


def make_inputs(name: str, *, seed: int, lengths, rows_per_request=None, row_len=None,
                H_i: int, D_i: int, H_q: int, D_k: int, D_v: int, k: int,
                softmax_scale: float, q_scale: float = 1.0,
                key_mode: str = "uniform", near_fraction: float = 0.1,
                n_distinct: int = 16) -> DecodeInputs:
    """Build a problem from its shape and distribution recipe.

    key_mode:
      ``uniform``       every key entry U{-8..7};
      ``near_parallel`` each position independently with probability
                        ``near_fraction`` takes ``q_idx[row, head 0] + U{-2..2}``
                        (the request's first query row), otherwise U{-8..7};
      ``distinct``      ``n_distinct`` vectors U{-8..7}; each position picks one
                        uniformly.
    """
    lengths = [int(x) for x in lengths]
    B = len(lengths)
    if rows_per_request is None:
        rows_per_request = [1] * B
    offsets = np.zeros(B + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(lengths)
    row_offsets = np.zeros(B + 1, dtype=np.int32)
    row_offsets[1:] = np.cumsum(rows_per_request)
    R = int(row_offsets[-1])
    L_total = int(offsets[-1])
    if row_len is None:
        rl = []
        for b in range(B):
            rl += [lengths[b]] * rows_per_request[b]
        row_len = np.asarray(rl, dtype=np.int32)
    row_len = np.asarray(row_len, dtype=np.int32)

    q_idx = uniform_nibbles(seed, TAG_Q_IDX, R * H_i * D_i).reshape(R, H_i, D_i)
    w_idx = uniform_int(seed, TAG_W_IDX, R * H_i, 1, 4).astype(np.int32).reshape(R, H_i)

    if key_mode == "distinct":
        vecs = uniform_nibbles(seed, TAG_DISTINCT_VEC, n_distinct * D_i).reshape(n_distinct, D_i)
        pick = uniform_int(seed, TAG_DISTINCT_PICK, L_total, 0, n_distinct - 1)
        k_idx = vecs[pick]
    else:
        k_idx = uniform_nibbles(seed, TAG_K_IDX, L_total * D_i).reshape(L_total, D_i)
        if key_mode == "near_parallel":
            near = bernoulli(seed, TAG_NEAR_PICK, L_total, near_fraction)
            noise = uniform_int(seed, TAG_NEAR_NOISE, L_total * D_i, -2, 2).reshape(L_total, D_i)
            for b in range(B):
                lo, hi = int(offsets[b]), int(offsets[b + 1])
                if rows_per_request[b] == 0 or hi == lo:
                    continue
                base = q_idx[row_offsets[b], 0].astype(np.int16)
                sel = np.nonzero(near[lo:hi])[0] + lo
                k_idx[sel] = (base[None, :] + noise[sel]).astype(np.int8)
        elif key_mode != "uniform":
            raise ValueError(key_mode)
    k_idx = np.ascontiguousarray(k_idx, dtype=np.int8)

    q = normal_bf16(seed, TAG_Q, R * H_q * D_k, q_scale).reshape(R, H_q, D_k)
    kv = normal_bf16(seed, TAG_KV, L_total * D_k).reshape(L_total, D_k)
    return DecodeInputs(name=name, R=R, B=B, H_i=H_i, D_i=D_i, H_q=H_q, D_k=D_k, D_v=D_v,
                        k=k, softmax_scale=float(softmax_scale), q_idx=q_idx, w_idx=w_idx,
                        k_idx=k_idx, q=q, kv=kv, offsets=offsets, row_offsets=row_offsets,
                        row_len=row_len)


# --- the five workloads -------------------------------------------------------

MLA = dict(H_i=64, D_i=128, H_q=64, D_k=576, D_v=512, k=2048, softmax_scale=1.0 / 24.0)


def tiny(layer: int = 0, L: int = 4096) -> DecodeInputs:
    """1 query, L=4096; q/k U{-8..7}, w U{1..4}; k=256; 8 heads, K=V width 64,
    queries N(0,1)/8 (the 1/sqrt(64) scale applied before bf16 rounding), so the
    kernel's softmax scale is 1."""
    return make_inputs("tiny", seed=config_seed(1, layer), lengths=[L], H_i=4, D_i=32,
                       H_q=8, D_k=64, D_v=64, k=256, softmax_scale=1.0, q_scale=0.125)


def l64k(layer: int = 0, L: int = 65536) -> DecodeInputs:
    return make_inputs("l64k", seed=config_seed(2, layer), lengths=[L],
                       key_mode="near_parallel", **MLA)


def l300k(layer: int = 0, L: int = 307200) -> DecodeInputs:
    return make_inputs("l300k", seed=config_seed(3, layer), lengths=[L],
                       key_mode="near_parallel", **MLA)


def batch32(B: int = 32, lo: int = 4096, hi: int = 131072, layer: int = 0,
            k: Optional[int] = None) -> DecodeInputs:
    seed = config_seed(4, layer)
    lengths = uniform_int(seed, TAG_LENGTHS, B, lo, hi)
    kw = dict(MLA)
    if k is not None:
        kw["k"] = k
    return make_inputs("batch32", seed=seed, lengths=lengths, key_mode="near_parallel", **kw)


def causal64(L: int = 131072, R: int = 64, layer: int = 0, k: Optional[int] = None) -> DecodeInputs:
    """R causal rows over one cache of L positions: row i sees L - R + i + 1."""
    row_len = np.arange(L - R + 1, L + 1, dtype=np.int32)
    kw = dict(MLA)
    if k is not None:
        kw["k"] = k
    return make_inputs("causal64", seed=config_seed(5, layer), lengths=[L],
                       rows_per_request=[R], row_len=row_len, key_mode="distinct", **kw)


def prefill(L: int = 10240, R: int = 2048, layer: int = 0, k: Optional[int] = None) -> DecodeInputs:
    """A prefill chunk: the last R positions of an L-position context are the
    chunk's query rows; row i sees L - R + i + 1 positions (causal).  Keys as
    ``l64k`` (10% near-parallel to the chunk's first query row)."""
    row_len = np.arange(L - R + 1, L + 1, dtype=np.int32)
    kw = dict(MLA)
    if k is not None:
        kw["k"] = k
    return make_inputs("prefill", seed=config_seed(6, layer), lengths=[L],
                       rows_per_request=[R], row_len=row_len, key_mode="near_parallel", **kw)


def fp8_cache(x: DecodeInputs, with_scale: bool = True) -> DecodeInputs:
    """The same problem over an FP8 E4M3 cache (codes uint8 [L_total, D_k] and
    float32 per-row scales), written from ``x.kv`` as described in the module
    docstring.  ``with_scale=False`` stores e4m3(kv) directly with no scales
    (kv_scale None, i.e. all 1; N(0,1) rows stay far inside e4m3's range)."""
    import torch

    bits = np.ascontiguousarray(x.kv, dtype=np.uint16)
    rows = torch.from_numpy((bits.astype(np.uint32) << np.uint32(16)).view(np.float32))
    if with_scale:
        amax = rows.abs().amax(dim=1) if rows.shape[1] else torch.zeros(rows.shape[0])
        scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        y = (rows / scale[:, None]).clamp(-448.0, 448.0)
        kv_scale = scale.numpy().astype(np.float32)
    else:
        y = rows.clamp(-448.0, 448.0)
        kv_scale = None
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return dataclasses.replace(x, name=x.name + "_fp8", kv=np.ascontiguousarray(codes),
                               kv_format="e4m3", kv_scale=kv_scale)


@dataclasses.dataclass
class FrontEndInputs:
    """Inputs of the indexer front end, host arrays only: ``x`` bf16 bits
    [R, d]; ``wq`` = (codes uint8 [H_i * D_i, d], scale bf16 bits [H_i * D_i, d/64],
    bias bf16 bits [H_i * D_i, d/64]); ``ww`` the same for [H_i, d]."""
    name: str
    R: int
    d: int
    H_i: int
    D_i: int
    x: np.ndarray
    wq: tuple
    ww: tuple


def _affine_weights(seed: int, which: int, O: int, d: int):
    g = d // 64
    codes = uniform_int(seed, TAG_FE_CODES + 3 * which, O * d, 0, 255).astype(np.uint8).reshape(O, d)
    s0 = np.sqrt(12.0) / (255.0 * np.sqrt(d))
    scale = s0 * uniform_int(seed, TAG_FE_SCALE + 3 * which, O * g, 192, 320).astype(np.float64) / 256.0
    scale_bits = f32_to_bf16_bits(scale.astype(np.float32))
    bias = -bf16_bits_to_f64(scale_bits) * uniform_int(seed, TAG_FE_BIAS + 3 * which, O * g, 120, 135)
    bias_bits = f32_to_bf16_bits(bias.astype(np.float32))
    return codes, scale_bits.reshape(O, g), bias_bits.reshape(O, g)


def front_end(R: int = 1, d: int = 6144, H_i: int = 64, D_i: int = 128, seed: int = 0x5EED) -> FrontEndInputs:
    """Seeded front-end inputs (see the module docstring); ``d`` a multiple of 64."""
    if d % 64:
        raise ValueError("d must be a multiple of 64 (the weight group)")
    x = normal_bf16(seed, TAG_FE_X, R * d).reshape(R, d)
    return FrontEndInputs(name=f"front_R{R}_d{d}", R=R, d=d, H_i=H_i, D_i=D_i, x=x,
                          wq=_affine_weights(seed, 0, H_i * D_i, d),
                          ww=_affine_weights(seed, 1, H_i, d))

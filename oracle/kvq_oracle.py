"""CPU oracle for quantized KV-cache decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference`` arm) use it.
It shares no code, table or helper with the CUDA path.

What it computes, and which passage each step follows
-----------------------------------------------------
Sources are the web pages this project is built from; each is cited by its
title and section.

* "KV Cache Quantization Analysis" (ryotta.opik.net, KV 캐시 양자화 심층 분석),
  section 2 "양자화 기초 / 핵심 개념": uniform (affine) quantization
  ``q = round(x/s + z)``, dequantization ``x_hat = s*(q - z)``; asymmetric
  (z != 0) when the distribution is off-centre; per-tensor / per-channel /
  per-token granularity.
* same page, section 3 "Key=per-channel, Value=per-token": Keys quantized per
  channel (over a group of tokens), Values per token; the most recent tokens
  kept in full precision as a sliding residual window.
* same page, section 4 "FP8 / INT8": the two OCP FP8 formats, E4M3
  (4 exponent, 3 mantissa bits) and E5M2 (5 exponent, 2 mantissa bits), each
  with an fp32 scale.
* same page, section 5 "구현·시스템 고려사항": quantize the new token's K,V
  right after they are computed, store them, dequantize right before attention.
* same page, closing box "메모리 크기 감각": ``KV_bytes = 2 * L * n_kv_heads *
  head_dim * seq_len * batch * bytes`` (bytes: FP16 2, FP8/INT8 1, INT4 0.5,
  INT2 0.25).
* "W4A16 + KV cache quantization combined accuracy" (hrletsgo.me), section
  "메모리 압박의 이중 구조": the Llama-3-70B worked example of the same
  formula (about 40 GB in bf16, 20 GB FP8, 10 GB INT4); section
  "오차가 어디서 만나는가": ``softmax(Q K^T / sqrt(d))``; section
  "어떤 레이어가 더 민감한가": the first (sink) token's K/V kept in 16-bit
  precision, FP8/INT8 on early and late layers and INT4 in the middle;
  section on the vLLM flags: the ``fp8_e5m2`` KV dtype and "skip layers"
  whose KV cache is left unquantized.

Readings where the pages leave a step open:

* scale and zero-point of a group come from its min m and max M:
  ``s = (M - m) / (2^b - 1)``, ``z = -(m / s)`` (float zero-point); a group
  whose ``s`` is not a normal positive float (constant group) uses ``s = 1``;
* every operation of the quantizer is one IEEE fp32 operation, rounded to
  nearest-even, with no fused multiply-add: ``x/s`` is a true division and
  ``round`` is round-half-to-even;
* FP8 is OCP E4M3FN (largest finite 448), round-to-nearest-even with
  saturation to +-448, the sign of zero kept; the per-tensor scale is
  ``amax / 448`` (``1`` when ``amax == 0``) of the tensor it calibrates;
* FP8 E5M2 is the OCP E5M2 format (IEEE-style: infinities and NaNs at the top
  exponent, largest finite 57344), encoded the same way (nearest, ties to the
  even code, saturating to +-57344) with the scale ``amax / 57344``;
* a "skip layer" (format ``bf16``) keeps every token's K and V in bf16: no
  quantized tokens, attention over the stored values;
* the cache keeps the first S tokens in bf16, quantizes tokens in groups of G
  once R + G tokens are waiting, so at least R recent tokens stay bf16
  (``Q_n = max(0, floor((T - S - R) / G)) * G``); FP8 uses G = 1, R = 0;
* attention is computed in fp64 on the dequantized values ``s*(q - z)``
  (also in fp64), ``lse = max + ln(sum exp(score - max))`` (natural log).
* pre-RoPE Keys ("KV Cache Quantization Analysis", section 3, the RoPE bullet:
  the rotation mixes channel pairs and smears the Key outliers, so KVQuant
  quantizes Keys before RoPE; section 4, KVQuant item (ii)): a layer with
  ``rope_base > 0`` stores its Keys as given (before the rotation) and attention
  rotates each dequantized Key at its own position t, rotate-half pairing
  ``(c, c + d/2)``, angle ``t * rope_base^(-2i/d)`` for pair i, in fp64; the
  query arrives already rotated at its own position.
* dense-and-sparse outliers (same page, section 4, KVQuant item (iv): outliers
  separated per vector; section 2: a few large values widen the grid and cost
  the other values their resolution): in a layer with ``k_outliers`` /
  ``v_outliers`` = n > 0, every quantized Key row and Value row keeps its n
  entries of largest magnitude (ties: the lower channel) exactly, as bf16, in a
  sparse list ordered by channel; the dense remainder, those entries set to 0,
  is quantized as usual (Keys per channel over the group, Values per token);
  the dequantized value is the dense one plus the sparse one.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

import numpy as np

F32 = np.float32
FLT_MIN = np.finfo(np.float32).tiny          # smallest normal fp32
E4M3_MAX = 448.0
E5M2_MAX = 57344.0


# --------------------------------------------------------------------------- #
# bf16 (how the inputs are stored)
# --------------------------------------------------------------------------- #


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- #
# C1 -- integer affine quantizer
# "KV Cache Quantization Analysis", section 2 (q = round(x/s + z), x_hat = s(q - z))
# --------------------------------------------------------------------------- #


def affine_quantize(x: np.ndarray, bits: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantize groups along the last axis of ``x`` (float32) to ``bits`` bits.

    Returns (codes uint8 with the shape of x, s float32, z float32) where s and z
    have the shape of x without its last axis.  Each group is asymmetric:
    its minimum maps to code 0 and its maximum to code 2^b - 1.
    """
    x = np.asarray(x, dtype=F32)
    levels = F32(2 ** bits - 1)
    lo = x.min(axis=-1)
    hi = x.max(axis=-1)
    s = (hi - lo) / levels                                   # fp32 subtract, fp32 divide
    s = np.where(s >= FLT_MIN, s, F32(1.0)).astype(F32)      # constant group -> s = 1
    z = (-(lo / s)).astype(F32)                              # float zero-point
    t = (x / s[..., None]).astype(F32)                       # true fp32 division
    t = (t + z[..., None]).astype(F32)                       # fp32 add
    q = np.rint(t)                                           # round half to even
    q = np.clip(q, 0, 2 ** bits - 1).astype(np.uint8)
    return q, s, z


def affine_dequantize_f32(codes: np.ndarray, s: np.ndarray, z: np.ndarray) -> np.ndarray:
    """x_hat = s * (q - z) evaluated as two fp32 operations (what the cache export returns)."""
    qf = codes.astype(F32)
    return (s * (qf - z).astype(F32)).astype(F32)


def affine_dequantize_f64(codes: np.ndarray, s: np.ndarray, z: np.ndarray) -> np.ndarray:
    """x_hat = s * (q - z) in fp64 (the value attention is defined on)."""
    return s.astype(np.float64) * (codes.astype(np.float64) - z.astype(np.float64))


# --------------------------------------------------------------------------- #
# C2 -- FP8 E4M3 ("KV Cache Quantization Analysis", section 4, FP8 / INT8)
# Encoder and decoder written from the OCP E4M3FN definition:
#   1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
#   subnormal (m * 2^-9); S.1111.111 is NaN; no infinities; max finite 448.
# --------------------------------------------------------------------------- #


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3FN code (uint8) -> float64 value (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.power(2.0, e - 7)
    sub = m * 2.0 ** -9
    mag = np.where(e == 0, sub, normal)
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


_E4M3_POS = e4m3_decode(np.arange(0, 0x7F))   # codes 0x00 .. 0x7E, increasing, 0 .. 448


def _encode_nearest(v: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """float32 values -> code of the nearest of the non-negative finite values
    ``pos`` (indexed by code, increasing), ties to the even code, magnitudes at
    or beyond the largest value saturating to it; the sign bit is the sign of
    the input (so -0.0 and small negatives give 0x80)."""
    v = np.asarray(v, dtype=F32).astype(np.float64)
    a = np.abs(v)
    idx = np.searchsorted(pos, a)                            # first value >= a
    idx = np.clip(idx, 1, len(pos) - 1)
    lo_c = idx - 1
    hi_c = idx
    d_lo = a - pos[lo_c]
    d_hi = pos[hi_c] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi_c % 2 == 0))
    mag = np.where(pick_hi, hi_c, lo_c)
    mag = np.where(a >= pos[-1], len(pos) - 1, mag)          # saturate (satfinite)
    mag = np.where(a <= pos[0], 0, mag)
    sign = np.signbit(v).astype(np.int64) << 7
    return (mag | sign).astype(np.uint8)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float32 values -> nearest E4M3FN code, ties to the even code, saturating at +-448."""
    return _encode_nearest(v, _E4M3_POS)


# E5M2 (same section; the OCP E5M2 definition): 1 sign bit, 5 exponent bits
# (bias 15), 2 mantissa bits; exponent field 0 is subnormal (m * 2^-16);
# exponent field 31 holds +-infinity (m = 0) and NaN; max finite 57344.


def e5m2_decode(codes: np.ndarray) -> np.ndarray:
    """E5M2 code (uint8) -> float64 value (+-inf, NaN for the top exponent)."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 2) & 0x1F
    m = c & 0x3
    normal = (1.0 + m / 4.0) * np.power(2.0, e - 15)
    sub = m * 2.0 ** -16
    mag = np.where(e == 0, sub, normal)
    mag = np.where(e == 0x1F, np.where(m == 0, np.inf, np.nan), mag)
    return sign * mag


_E5M2_POS = e5m2_decode(np.arange(0, 0x7C))   # codes 0x00 .. 0x7B, increasing, 0 .. 57344


def e5m2_encode(v: np.ndarray) -> np.ndarray:
    """float32 values -> nearest finite E5M2 code, ties to the even code, saturating at +-57344."""
    return _encode_nearest(v, _E5M2_POS)


FP8_FORMATS = {"fp8_e4m3": (e4m3_encode, e4m3_decode, E4M3_MAX),
               "fp8_e5m2": (e5m2_encode, e5m2_decode, E5M2_MAX)}


def fp8_decode(codes: np.ndarray, fmt: str = "fp8_e4m3") -> np.ndarray:
    return FP8_FORMATS[fmt][1](codes)


def fp8_tensor_scale(x: np.ndarray, fmt: str = "fp8_e4m3") -> np.float32:
    """Per-tensor fp32 scale amax / (largest finite value of the format) of a
    calibration tensor (1 when amax == 0): 448 for E4M3, 57344 for E5M2."""
    amax = F32(np.max(np.abs(np.asarray(x, dtype=F32)))) if np.size(x) else F32(0.0)
    if amax == 0:
        return F32(1.0)
    return F32(amax / F32(FP8_FORMATS[fmt][2]))


def fp8_quantize(x: np.ndarray, s: np.float32, fmt: str = "fp8_e4m3") -> np.ndarray:
    """code = FP8(fl32(x / s)) in the given format."""
    return FP8_FORMATS[fmt][0]((np.asarray(x, dtype=F32) / F32(s)).astype(F32))


# --------------------------------------------------------------------------- #
# C3 -- the cache of one (layer, sequence, kv head)
# "KV Cache Quantization Analysis", sections 3 (residual window) and 5
# (quantize on write); "W4A16 + KV ..." (sink token kept in 16-bit precision)
# --------------------------------------------------------------------------- #


@dataclasses.dataclass(frozen=True)
class Spec:
    fmt: str          # "int2" | "int4" | "int8" | "fp8_e4m3" | "fp8_e5m2" | "bf16"
    d: int = 128
    G: int = 32       # Key group (tokens); 1 for FP8; unused for bf16
    Gv: int = 128     # Value group (channels)
    R: int = 0        # residual window (bf16)
    S: int = 0        # sink tokens (bf16)
    rope_base: float = 0.0  # > 0: Keys stored before RoPE, rotated at their position by attention
    k_outliers: int = 0     # per quantized Key row: entries kept apart (sparse, bf16)
    v_outliers: int = 0     # per quantized Value row

    @property
    def bits(self) -> int:
        return {"int2": 2, "int4": 4, "int8": 8, "fp8_e4m3": 8, "fp8_e5m2": 8, "bf16": 16}[self.fmt]

    @property
    def is_fp8(self) -> bool:
        return self.fmt in FP8_FORMATS

    @property
    def is_bf16(self) -> bool:
        """A skip layer: nothing is quantized, every token stays bf16."""
        return self.fmt == "bf16"


def token_split(T: int, spec: Spec) -> Tuple[int, int, int]:
    """(sink tokens, quantized tokens Q_n, residual tokens r) of a cache holding T tokens."""
    n_sink = min(T, spec.S)
    n = T - n_sink
    if spec.is_fp8:
        return n_sink, n, 0
    if spec.is_bf16:
        return n_sink, 0, n
    qn = max(0, (n - spec.R) // spec.G) * spec.G
    return n_sink, qn, n - qn


@dataclasses.dataclass
class HeadCache:
    """Logical (layout-free) cache of one (layer, sequence, kv head).

    sink_k/v, resid_k/v: bf16 values as float32 [n, d].
    k_codes, v_codes: uint8 [Q_n, d] (one code per element).
    INT: k_s, k_z [Q_n/G, d]; v_s, v_z [Q_n, d/Gv].
    FP8: k_scale, v_scale (per tensor).
    """

    spec: Spec
    sink_k: np.ndarray
    sink_v: np.ndarray
    k_codes: np.ndarray
    v_codes: np.ndarray
    resid_k: np.ndarray
    resid_v: np.ndarray
    k_s: Optional[np.ndarray] = None
    k_z: Optional[np.ndarray] = None
    v_s: Optional[np.ndarray] = None
    v_z: Optional[np.ndarray] = None
    k_scale: Optional[np.float32] = None
    v_scale: Optional[np.float32] = None
    # dense-and-sparse: per quantized row, the outliers' channels (ascending) and bf16 values
    k_sp_idx: Optional[np.ndarray] = None   # int64 [Q_n, k_outliers]
    k_sp_val: Optional[np.ndarray] = None   # float32 [Q_n, k_outliers]
    v_sp_idx: Optional[np.ndarray] = None
    v_sp_val: Optional[np.ndarray] = None

    @property
    def T(self) -> int:
        return len(self.sink_k) + len(self.k_codes) + len(self.resid_k)


def split_outliers(x: np.ndarray, n: int):
    """Dense-and-sparse split of rows x [m, d]: the n entries of largest magnitude of each row
    (ties: the lower channel) leave it.  Returns (dense: x with them set to 0, idx [m, n] ascending,
    val [m, n]: their values)."""
    x = np.asarray(x, dtype=F32)
    m, d = x.shape
    if n == 0:
        return x.copy(), np.zeros((m, 0), np.int64), np.zeros((m, 0), F32)
    order = np.lexsort((np.arange(d)[None, :].repeat(m, 0), -np.abs(x)), axis=1)  # by |x| desc, then channel
    idx = np.sort(order[:, :n], axis=1)
    val = np.take_along_axis(x, idx, axis=1)
    dense = x.copy()
    np.put_along_axis(dense, idx, F32(0.0), axis=1)
    return dense, idx, val


def quantize_key_groups(k: np.ndarray, spec: Spec):
    """Keys per channel: every channel of every G-token group is one quantization group (of the
    dense part when the layer keeps outliers apart).  Returns codes, s, z, sparse idx, sparse val."""
    qn, d = k.shape
    k, sp_idx, sp_val = split_outliers(k, spec.k_outliers)
    g = k.reshape(qn // spec.G, spec.G, d).transpose(0, 2, 1)    # [groups, d, G]
    codes, s, z = affine_quantize(g, spec.bits)
    return codes.transpose(0, 2, 1).reshape(qn, d), s, z, sp_idx, sp_val   # s, z: [groups, d]


def quantize_value_tokens(v: np.ndarray, spec: Spec):
    """Values per token: every Gv-channel slice of every token is one quantization group (of the
    dense part when the layer keeps outliers apart).  Returns codes, s, z, sparse idx, sparse val."""
    qn, d = v.shape
    v, sp_idx, sp_val = split_outliers(v, spec.v_outliers)
    g = v.reshape(qn, d // spec.Gv, spec.Gv)
    codes, s, z = affine_quantize(g, spec.bits)
    return codes.reshape(qn, d), s, z, sp_idx, sp_val            # s, z: [Q_n, d/Gv]


def build_head_cache(k: np.ndarray, v: np.ndarray, spec: Spec,
                     k_scale: Optional[float] = None, v_scale: Optional[float] = None) -> HeadCache:
    """State of the cache after the tokens of ``k``, ``v`` (float32 [T, d], bf16 values) were written.

    Equal to T single-token appends (checked by ``append_token``).
    """
    T = k.shape[0]
    n_sink, qn, r = token_split(T, spec)
    q0, q1 = n_sink, n_sink + qn
    hc = HeadCache(spec, k[:n_sink].copy(), v[:n_sink].copy(), None, None, k[q1:].copy(), v[q1:].copy())
    if spec.is_fp8:
        hc.k_scale, hc.v_scale = F32(k_scale), F32(v_scale)
        hc.k_codes = fp8_quantize(k[q0:q1], hc.k_scale, spec.fmt)
        hc.v_codes = fp8_quantize(v[q0:q1], hc.v_scale, spec.fmt)
    elif spec.is_bf16:
        hc.k_codes = np.zeros((0, spec.d), np.uint8)
        hc.v_codes = np.zeros((0, spec.d), np.uint8)
    else:
        hc.k_codes, hc.k_s, hc.k_z, hc.k_sp_idx, hc.k_sp_val = quantize_key_groups(k[q0:q1], spec)
        hc.v_codes, hc.v_s, hc.v_z, hc.v_sp_idx, hc.v_sp_val = quantize_value_tokens(v[q0:q1], spec)
    return hc


def empty_head_cache(spec: Spec, k_scale=None, v_scale=None) -> HeadCache:
    d = spec.d
    z = np.zeros((0, d), F32)
    hc = HeadCache(spec, z.copy(), z.copy(), np.zeros((0, d), np.uint8), np.zeros((0, d), np.uint8),
                   z.copy(), z.copy())
    if spec.is_fp8:
        hc.k_scale, hc.v_scale = F32(k_scale), F32(v_scale)
    elif not spec.is_bf16:
        hc.k_s = np.zeros((0, d), F32)
        hc.k_z = np.zeros((0, d), F32)
        hc.v_s = np.zeros((0, d // spec.Gv), F32)
        hc.v_z = np.zeros((0, d // spec.Gv), F32)
        hc.k_sp_idx, hc.k_sp_val = np.zeros((0, spec.k_outliers), np.int64), np.zeros((0, spec.k_outliers), F32)
        hc.v_sp_idx, hc.v_sp_val = np.zeros((0, spec.v_outliers), np.int64), np.zeros((0, spec.v_outliers), F32)
    return hc


def append_token(hc: HeadCache, k_tok: np.ndarray, v_tok: np.ndarray) -> None:
    """Write one new token, following the quantize-on-write step.

    Sink slots fill first.  Otherwise the token joins the bf16 residual window;
    once R + G tokens wait there, the oldest G are quantized together (one Key
    group, G Value tokens) and leave the window.  FP8 quantizes at once.
    """
    spec = hc.spec
    k_tok = np.asarray(k_tok, F32).reshape(1, -1)
    v_tok = np.asarray(v_tok, F32).reshape(1, -1)
    if len(hc.sink_k) < spec.S:
        hc.sink_k = np.concatenate([hc.sink_k, k_tok])
        hc.sink_v = np.concatenate([hc.sink_v, v_tok])
        return
    if spec.is_fp8:
        hc.k_codes = np.concatenate([hc.k_codes, fp8_quantize(k_tok, hc.k_scale, spec.fmt)])
        hc.v_codes = np.concatenate([hc.v_codes, fp8_quantize(v_tok, hc.v_scale, spec.fmt)])
        return
    hc.resid_k = np.concatenate([hc.resid_k, k_tok])
    hc.resid_v = np.concatenate([hc.resid_v, v_tok])
    if not spec.is_bf16 and len(hc.resid_k) == spec.R + spec.G:
        kc, ks, kz, ki, kv = quantize_key_groups(hc.resid_k[:spec.G], spec)
        vc, vs, vz, vi, vv = quantize_value_tokens(hc.resid_v[:spec.G], spec)
        hc.k_sp_idx, hc.k_sp_val = np.concatenate([hc.k_sp_idx, ki]), np.concatenate([hc.k_sp_val, kv])
        hc.v_sp_idx, hc.v_sp_val = np.concatenate([hc.v_sp_idx, vi]), np.concatenate([hc.v_sp_val, vv])
        hc.k_codes = np.concatenate([hc.k_codes, kc])
        hc.k_s = np.concatenate([hc.k_s, ks])
        hc.k_z = np.concatenate([hc.k_z, kz])
        hc.v_codes = np.concatenate([hc.v_codes, vc])
        hc.v_s = np.concatenate([hc.v_s, vs])
        hc.v_z = np.concatenate([hc.v_z, vz])
        hc.resid_k = hc.resid_k[spec.G:]
        hc.resid_v = hc.resid_v[spec.G:]


def dequantized_f64(hc: HeadCache) -> Tuple[np.ndarray, np.ndarray]:
    """All T tokens' (k_hat, v_hat) in fp64, in token order [T, d]."""
    spec = hc.spec
    if spec.is_fp8:
        kq = float(hc.k_scale) * fp8_decode(hc.k_codes, spec.fmt)
        vq = float(hc.v_scale) * fp8_decode(hc.v_codes, spec.fmt)
    elif spec.is_bf16:
        kq = vq = np.zeros((0, spec.d))
    else:
        gk = np.repeat(np.arange(len(hc.k_s)), spec.G)
        kq = affine_dequantize_f64(hc.k_codes, hc.k_s[gk], hc.k_z[gk])
        vs = np.repeat(hc.v_s, spec.Gv, axis=1)
        vz = np.repeat(hc.v_z, spec.Gv, axis=1)
        vq = affine_dequantize_f64(hc.v_codes, vs, vz)
        # dense-and-sparse: the kept outliers add to the dense values at their channels
        rows = np.arange(kq.shape[0])[:, None]
        if spec.k_outliers:
            kq[rows, hc.k_sp_idx] += hc.k_sp_val.astype(np.float64)
        if spec.v_outliers:
            vq[rows, hc.v_sp_idx] += hc.v_sp_val.astype(np.float64)
    k = np.concatenate([hc.sink_k.astype(np.float64), kq, hc.resid_k.astype(np.float64)])
    v = np.concatenate([hc.sink_v.astype(np.float64), vq, hc.resid_v.astype(np.float64)])
    return k, v


def dequantized_f32(hc: HeadCache) -> Tuple[np.ndarray, np.ndarray]:
    """All T tokens' x_hat as the cache export defines it: fp32 ``s*(q - z)`` or ``s*fp8(q)``."""
    spec = hc.spec
    if spec.is_fp8:
        kq = (hc.k_scale * fp8_decode(hc.k_codes, spec.fmt).astype(F32)).astype(F32)
        vq = (hc.v_scale * fp8_decode(hc.v_codes, spec.fmt).astype(F32)).astype(F32)
    elif spec.is_bf16:
        kq = vq = np.zeros((0, spec.d), F32)
    else:
        gk = np.repeat(np.arange(len(hc.k_s)), spec.G)
        kq = affine_dequantize_f32(hc.k_codes, hc.k_s[gk], hc.k_z[gk])
        vs = np.repeat(hc.v_s, spec.Gv, axis=1)
        vz = np.repeat(hc.v_z, spec.Gv, axis=1)
        vq = affine_dequantize_f32(hc.v_codes, vs, vz)
        # dense-and-sparse: one more fp32 add at each kept outlier's channel
        rows = np.arange(kq.shape[0])[:, None]
        if spec.k_outliers:
            kq[rows, hc.k_sp_idx] = (kq[rows, hc.k_sp_idx] + hc.k_sp_val).astype(F32)
        if spec.v_outliers:
            vq[rows, hc.v_sp_idx] = (vq[rows, hc.v_sp_idx] + hc.v_sp_val).astype(F32)
    k = np.concatenate([hc.sink_k, kq, hc.resid_k]).astype(F32)
    v = np.concatenate([hc.sink_v, vq, hc.resid_v]).astype(F32)
    return k, v


# --------------------------------------------------------------------------- #
# pre-RoPE Keys ("KV Cache Quantization Analysis", section 3 RoPE bullet; section 4 KVQuant (ii))
# --------------------------------------------------------------------------- #


def rope_angles(positions: np.ndarray, d: int, base: float) -> np.ndarray:
    """Angles [len(positions), d/2] in fp64: position t times base^(-2i/d) for pair i."""
    inv_freq = np.power(float(base), -np.arange(0, d, 2, dtype=np.float64) / d)
    return np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope_rotate(x: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half RoPE of rows x [n, d] at the given positions, in fp64: channel pair
    (i, i + d/2) turned by the angle of pair i (x_i cos - x_{i+d/2} sin, x_{i+d/2} cos + x_i sin)."""
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    a = rope_angles(positions, x.shape[-1], base)
    c, s_ = np.cos(a), np.sin(a)
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s_, hi * c + lo * s_], axis=-1)


def attention_keys(hc: HeadCache) -> Tuple[np.ndarray, np.ndarray]:
    """(Keys, Values) in fp64 as attention sees them: the dequantized cache, the Keys
    rotated at their positions 0 .. T-1 when the layer stores them before RoPE."""
    k, v = dequantized_f64(hc)
    if hc.spec.rope_base > 0:
        k = rope_rotate(k, np.arange(k.shape[0]), hc.spec.rope_base)
    return k, v


# --------------------------------------------------------------------------- #
# C4 -- decode attention, softmax(q K^T / sqrt(d)) V, in fp64
# "W4A16 + KV ...", section "오차가 어디서 만나는가" (score formula)
# --------------------------------------------------------------------------- #


def attend_head(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, softmax_scale: float):
    """One query vector against T dequantized tokens.  Returns (out [d], lse)."""
    if k_hat.shape[0] == 0:
        return np.zeros(q.shape[-1]), -math.inf
    sigma = (k_hat @ np.asarray(q, np.float64)) * softmax_scale
    mu = sigma.max()
    e = np.exp(sigma - mu)
    ell = e.sum()
    out = (e @ v_hat) / ell
    return out, mu + math.log(ell)


def decode_attention(q: np.ndarray, caches: List[List[HeadCache]], softmax_scale: Optional[float] = None):
    """Decode step for a batch.

    q: [B, Hq, d] (float32 values of the bf16 queries); caches[b][h] for kv head h.
    Query head hq reads kv head hq // (Hq / Hkv) (grouped-query attention).
    Returns out [B, Hq, d] float64, lse [B, Hq] float64.
    """
    B, Hq, d = q.shape
    Hkv = len(caches[0])
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else softmax_scale
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        for h in range(Hkv):
            k_hat, v_hat = attention_keys(caches[b][h])
            for j in range(g):
                hq = h * g + j
                out[b, hq], lse[b, hq] = attend_head(q[b, hq], k_hat, v_hat, scale)
    return out, lse


def decode_attention_multi(q: np.ndarray, caches: List[List[HeadCache]], softmax_scale: Optional[float] = None):
    """Several new query tokens per sequence, each attending causally.

    The same score formula ("W4A16 + KV ...", section "오차가 어디서 만나는가")
    for M query tokens per sequence whose K, V are already the cache's last M
    tokens: query token i of a sequence with T cached tokens sits at position
    T - M + i and attends to tokens 0 .. T - M + i of the cache (as dequantized
    with all T tokens written).  q: [B, M, Hq, d].  Returns out [B, M, Hq, d],
    lse [B, M, Hq] (a query with no visible token: out 0, lse -inf).
    """
    B, M, Hq, d = q.shape
    Hkv = len(caches[0])
    g = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else softmax_scale
    out = np.zeros((B, M, Hq, d))
    lse = np.zeros((B, M, Hq))
    for b in range(B):
        for h in range(Hkv):
            k_hat, v_hat = attention_keys(caches[b][h])
            T = k_hat.shape[0]
            for i in range(M):
                n = max(0, T - M + i + 1)
                for j in range(g):
                    hq = h * g + j
                    out[b, i, hq], lse[b, i, hq] = attend_head(q[b, i, hq], k_hat[:n], v_hat[:n], scale)
    return out, lse


# --------------------------------------------------------------------------- #
# Byte accounting ("KV Cache Quantization Analysis", box "메모리 크기 감각")
# --------------------------------------------------------------------------- #


def kv_cache_bytes(layers: int, kv_heads: int, head_dim: int, seq_len: int, batch: int,
                   bytes_per_element: float) -> float:
    """KV_bytes = 2 (K and V) * L * n_kv_heads * head_dim * seq_len * batch * bytes."""
    return 2 * layers * kv_heads * head_dim * seq_len * batch * bytes_per_element


def block_format_bits_per_element(bits: int, block: int, scale_bits: int, zero_bits: int = 0) -> float:
    """Storage bits per element of a block format: ``bits`` per code plus one scale
    (and optional zero-point) per ``block`` elements."""
    return bits + (scale_bits + zero_bits) / block

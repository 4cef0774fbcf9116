"""Thin Python binding of libkvq (the C ABI in include/kvq.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of libkvq.so.  PyTorch is used for device memory and streams.  If the
library is missing, importing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kvq.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libkvq.so not found at {LIB_PATH}: build it first "
                      "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p
c_sz = ctypes.c_size_t

KVQ_OK = 0
STATUS = {0: "KVQ_OK", -1: "KVQ_ERR_INVALID_ARG", -2: "KVQ_ERR_UNSUPPORTED", -3: "KVQ_ERR_CUDA",
          -4: "KVQ_ERR_WORKSPACE"}
DEV_BAD_BLOCK, DEV_CAPACITY, DEV_TIMEOUT = 0x1, 0x2, 0x4
FORMATS = {"bf16": 1, "int2": 2, "int4": 4, "int8": 8, "fp8_e4m3": 16, "fp8_e5m2": 17}
FP8_FORMATS = (FORMATS["fp8_e4m3"], FORMATS["fp8_e5m2"])
FIELDS = ["qstore", "block_pool", "resid_k", "resid_v", "sink_k", "sink_v"]


class KvqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({status_string(status)})")
        self.status = status


class LayerConfig(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("num_kv_heads", "head_dim", "format", "k_group_tokens", "v_group_dims",
                                     "residual_tokens", "sink_tokens", "paged", "block_tokens", "capacity_tokens",
                                     "num_blocks", "max_blocks_per_seq")] + [("rope_base", ctypes.c_float),
                                                                             ("k_outliers", c_i32), ("v_outliers", c_i32)]


class LayerCache(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("qstore", "block_pool", "block_table", "resid_k", "resid_v", "sink_k", "sink_v",
                                    "k_tensor_scale", "v_tensor_scale")]


_P = ctypes.POINTER
_lib.kvq_cache_layout.argtypes = [_P(LayerConfig), c_i32, _P(c_sz)]
_lib.kvq_fp8_calibrate.argtypes = [c_vp, c_sz, c_vp, c_vp]
_lib.kvq_fp8_calibrate_format.argtypes = [c_vp, c_sz, c_i32, c_vp, c_vp]
_lib.kvq_quantize_append.argtypes = [_P(LayerConfig), _P(LayerCache), c_vp, c_vp, c_i32, c_vp, c_i32, c_vp, c_vp]
_lib.kvq_decode_workspace_size.argtypes = [_P(LayerConfig), c_i32, c_i32, _P(c_sz)]
_lib.kvq_decode_attention.argtypes = [_P(LayerConfig), _P(LayerCache), c_vp, c_i32, c_vp, c_i32, ctypes.c_float,
                                      c_vp, c_i32, c_vp, c_vp, c_sz, c_vp, c_vp]
_lib.kvq_decode_attention_multi.argtypes = [_P(LayerConfig), _P(LayerCache), c_vp, c_i32, c_i32, c_vp, c_i32,
                                            ctypes.c_float, c_vp, c_i32, c_vp, c_vp, c_sz, c_vp, c_vp]
_lib.kvq_append_decode_attention.argtypes = [_P(LayerConfig), _P(LayerCache), c_vp, c_vp, c_vp, c_i32, c_vp,
                                             c_i32, ctypes.c_float, c_vp, c_i32, c_vp, c_vp, c_sz, c_vp, c_vp]
_lib.kvq_decode_workspace_size_multi.argtypes = [_P(LayerConfig), c_i32, c_i32, c_i32, _P(c_sz)]
_lib.kvq_selftest_bounded_wait.argtypes = [_P(LayerConfig), _P(LayerCache), c_vp, c_i32, c_vp, c_i32, ctypes.c_float,
                                           c_vp, c_i32, c_vp, c_vp, c_sz, c_vp, c_vp]
_lib.kvq_lse_merge.argtypes = [c_vp, c_vp, c_i32, ctypes.c_int64, c_vp, c_i32, c_vp, c_vp]
_lib.kvq_decode_partials.argtypes = [_P(LayerConfig), _P(LayerCache), c_vp, c_i32, c_vp, c_i32, ctypes.c_float,
                                     c_vp, c_sz, c_vp, c_vp]
_lib.kvq_decode_combine.argtypes = [_P(LayerConfig), c_i32, c_i32, c_vp, c_i32, c_vp, c_vp, c_sz, c_vp]
_lib.kvq_decode_attention_static_scratch.argtypes = [_P(LayerConfig), _P(LayerCache), c_vp, c_i32, c_vp, c_i32,
                                                     ctypes.c_float, c_vp, c_i32, c_vp, c_vp, c_vp]
_lib.kvq_dequantize.argtypes = [_P(LayerConfig), _P(LayerCache), c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp]
_lib.kvq_status_string.argtypes = [c_i32]
_lib.kvq_status_string.restype = ctypes.c_char_p
for _fn in ("kvq_cache_layout", "kvq_fp8_calibrate", "kvq_fp8_calibrate_format", "kvq_quantize_append",
            "kvq_decode_workspace_size",
            "kvq_decode_attention", "kvq_decode_partials", "kvq_decode_combine", "kvq_dequantize",
            "kvq_decode_attention_multi", "kvq_decode_workspace_size_multi", "kvq_lse_merge",
            "kvq_selftest_bounded_wait",
            "kvq_decode_attention_static_scratch", "kvq_append_decode_attention"):
    getattr(_lib, _fn).restype = c_i32


def declared_symbols() -> Sequence[str]:
    """Entry points declared in include/kvq.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:kvq_status|const char\*)\s+(kvq_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return _lib.kvq_status_string(status).decode()


def _check(fn: str, st: int):
    if st != KVQ_OK:
        raise KvqError(fn, st)


def _ptr(t) -> Optional[int]:
    """Device (or host) address of a tensor, an int, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(fmt: str, num_kv_heads: int, G: int, Gv: int, R: int, S: int, *, paged: bool = False,
                block_tokens: int = 0, capacity_tokens: int = 0, num_blocks: int = 0,
                max_blocks_per_seq: int = 0, head_dim: int = 128, rope_base: float = 0.0, k_outliers: int = 0,
                v_outliers: int = 0) -> LayerConfig:
    """rope_base > 0: the layer's Keys are appended before RoPE and rotated at their position by the decode.
    k_outliers / v_outliers > 0: dense-and-sparse rows (that many entries per row kept exactly)."""
    return LayerConfig(num_kv_heads, head_dim, FORMATS[fmt], G, Gv, R, S, int(paged), block_tokens,
                       capacity_tokens, num_blocks, max_blocks_per_seq, rope_base, k_outliers, v_outliers)


def cache_layout(cfg: LayerConfig, num_seqs: int) -> Dict[str, int]:
    out = (c_sz * len(FIELDS))()
    _check("kvq_cache_layout", _lib.kvq_cache_layout(ctypes.byref(cfg), num_seqs, out))
    return {n: int(out[i]) for i, n in enumerate(FIELDS)}


def fp8_calibrate(x, n: int, scale_out, stream=None, fmt: str = "fp8_e4m3") -> None:
    """Per-tensor FP8 scale amax / (448 for E4M3, 57344 for E5M2) of n bf16 values, on the device."""
    if fmt == "fp8_e4m3":
        _check("kvq_fp8_calibrate", _lib.kvq_fp8_calibrate(_ptr(x), n, _ptr(scale_out), _stream_ptr(stream)))
    else:
        _check("kvq_fp8_calibrate_format",
               _lib.kvq_fp8_calibrate_format(_ptr(x), n, FORMATS[fmt], _ptr(scale_out), _stream_ptr(stream)))


def quantize_append(cfg: LayerConfig, cache: LayerCache, k_new, v_new, n_new: int, seq_lens, batch: int,
                    dev_status=None, stream=None) -> None:
    """Write n_new tokens per (sequence, kv head): sink, bf16 window, quantized spills."""
    _check("kvq_quantize_append",
           _lib.kvq_quantize_append(ctypes.byref(cfg), ctypes.byref(cache), _ptr(k_new), _ptr(v_new), n_new,
                                    _ptr(seq_lens), batch, _ptr(dev_status), _stream_ptr(stream)))


def decode_workspace_size(cfg: LayerConfig, batch: int, num_q_heads: int) -> int:
    out = c_sz(0)
    _check("kvq_decode_workspace_size",
           _lib.kvq_decode_workspace_size(ctypes.byref(cfg), batch, num_q_heads, ctypes.byref(out)))
    return int(out.value)


def decode_attention(cfg: LayerConfig, cache: LayerCache, q, num_q_heads: int, seq_lens, batch: int,
                     softmax_scale: float, out, out_bf16: bool, lse, workspace, workspace_bytes: int,
                     dev_status=None, stream=None) -> None:
    """One decode step of attention over the cache (fused split pass + log-sum-exp merge)."""
    _check("kvq_decode_attention",
           _lib.kvq_decode_attention(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), num_q_heads, _ptr(seq_lens),
                                     batch, softmax_scale, _ptr(out), int(out_bf16), _ptr(lse), _ptr(workspace),
                                     workspace_bytes, _ptr(dev_status), _stream_ptr(stream)))


def append_decode_attention(cfg: LayerConfig, cache: LayerCache, k_new, v_new, seq_lens, batch: int, q,
                            num_q_heads: int, softmax_scale: float, out, out_bf16: bool, lse, workspace,
                            workspace_bytes: int, dev_status=None, stream=None) -> None:
    """One whole decode step: append one token per sequence (seq_lens: lengths before it), then attention."""
    _check("kvq_append_decode_attention",
           _lib.kvq_append_decode_attention(ctypes.byref(cfg), ctypes.byref(cache), _ptr(k_new), _ptr(v_new),
                                            _ptr(seq_lens), batch, _ptr(q), num_q_heads, softmax_scale, _ptr(out),
                                            int(out_bf16), _ptr(lse), _ptr(workspace), workspace_bytes,
                                            _ptr(dev_status), _stream_ptr(stream)))


def decode_workspace_size_multi(cfg: LayerConfig, batch: int, n_query: int, num_q_heads: int) -> int:
    """Workspace bytes of decode_attention_multi (kvq_decode_workspace_size_multi)."""
    out = c_sz(0)
    _check("kvq_decode_workspace_size_multi",
           _lib.kvq_decode_workspace_size_multi(ctypes.byref(cfg), batch, n_query, num_q_heads, ctypes.byref(out)))
    return int(out.value)


def decode_attention_multi(cfg: LayerConfig, cache: LayerCache, q, n_query: int, num_q_heads: int, seq_lens,
                           batch: int, softmax_scale: float, out, out_bf16: bool, lse, workspace, workspace_bytes: int,
                           dev_status=None, stream=None) -> None:
    """n_query causal query tokens per sequence in one launch; q, out: [B][n_query][Hq][d]."""
    _check("kvq_decode_attention_multi",
           _lib.kvq_decode_attention_multi(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), n_query, num_q_heads,
                                           _ptr(seq_lens), batch, softmax_scale, _ptr(out), int(out_bf16), _ptr(lse),
                                           _ptr(workspace), workspace_bytes, _ptr(dev_status), _stream_ptr(stream)))


def selftest_bounded_wait(cfg: LayerConfig, cache: LayerCache, q, num_q_heads: int, seq_lens, batch: int,
                          softmax_scale: float, out, out_bf16: bool, lse, workspace, workspace_bytes: int, dev_status,
                          stream=None) -> None:
    """Decode with one bulk copy withheld: must report DEV_TIMEOUT in dev_status and finish."""
    _check("kvq_selftest_bounded_wait",
           _lib.kvq_selftest_bounded_wait(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), num_q_heads,
                                          _ptr(seq_lens), batch, softmax_scale, _ptr(out), int(out_bf16), _ptr(lse),
                                          _ptr(workspace), workspace_bytes, _ptr(dev_status), _stream_ptr(stream)))


def lse_merge(o_parts, lse_parts, n_parts: int, rows: int, out, out_bf16: bool, lse_out=None, stream=None) -> None:
    """Merge per-part (out, lse) rows over disjoint token parts; o_parts [n][rows][128] fp32."""
    _check("kvq_lse_merge", _lib.kvq_lse_merge(_ptr(o_parts), _ptr(lse_parts), n_parts, rows, _ptr(out), int(out_bf16),
                                               _ptr(lse_out), _stream_ptr(stream)))


def decode_partials(cfg: LayerConfig, cache: LayerCache, q, num_q_heads: int, seq_lens, batch: int,
                    softmax_scale: float, workspace, workspace_bytes: int, dev_status=None, stream=None) -> None:
    _check("kvq_decode_partials",
           _lib.kvq_decode_partials(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), num_q_heads, _ptr(seq_lens),
                                    batch, softmax_scale, _ptr(workspace), workspace_bytes, _ptr(dev_status),
                                    _stream_ptr(stream)))


def decode_combine(cfg: LayerConfig, num_q_heads: int, batch: int, out, out_bf16: bool, lse, workspace,
                   workspace_bytes: int, stream=None) -> None:
    _check("kvq_decode_combine",
           _lib.kvq_decode_combine(ctypes.byref(cfg), num_q_heads, batch, _ptr(out), int(out_bf16), _ptr(lse),
                                   _ptr(workspace), workspace_bytes, _stream_ptr(stream)))


def decode_attention_static_scratch(cfg: LayerConfig, cache: LayerCache, q, num_q_heads: int, seq_lens, batch: int,
                                    softmax_scale: float, out, out_bf16: bool, lse, dev_status=None,
                                    stream=None) -> None:
    """Decode attention using the library's fixed device scratch instead of a workspace (allocates nothing)."""
    _check("kvq_decode_attention_static_scratch",
           _lib.kvq_decode_attention_static_scratch(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), num_q_heads,
                                                    _ptr(seq_lens), batch, softmax_scale, _ptr(out), int(out_bf16),
                                                    _ptr(lse), _ptr(dev_status), _stream_ptr(stream)))


def dequantize(cfg: LayerConfig, cache: LayerCache, seq_lens, batch: int, max_tokens: int, k_out, v_out,
               dev_status=None, stream=None) -> None:
    _check("kvq_dequantize",
           _lib.kvq_dequantize(ctypes.byref(cfg), ctypes.byref(cache), _ptr(seq_lens), batch, max_tokens,
                               _ptr(k_out), _ptr(v_out), _ptr(dev_status), _stream_ptr(stream)))


# --------------------------------------------------------------------------- #
# Device buffers of one layer's cache (allocation through PyTorch)
# --------------------------------------------------------------------------- #


class CacheLayer:
    """The device buffers of one layer's quantized cache for ``num_seqs`` sequences."""

    def __init__(self, cfg: LayerConfig, num_seqs: int, device="cuda", zero: bool = True):
        import torch
        self.cfg = cfg
        self.num_seqs = num_seqs
        self.sizes = cache_layout(cfg, num_seqs)
        alloc = torch.zeros if zero else torch.empty
        self.buf = {n: (alloc(s, dtype=torch.uint8, device=device) if s else None) for n, s in self.sizes.items()}
        self.block_table = None
        if cfg.paged:
            self.block_table = torch.full((num_seqs, cfg.max_blocks_per_seq), -1, dtype=torch.int32, device=device)
        self.k_tensor_scale = self.v_tensor_scale = None
        if cfg.format in FP8_FORMATS:
            self.k_tensor_scale = torch.ones(1, dtype=torch.float32, device=device)
            self.v_tensor_scale = torch.ones(1, dtype=torch.float32, device=device)

    def struct(self) -> LayerCache:
        c = LayerCache()
        for n in FIELDS:
            setattr(c, n, _ptr(self.buf[n]))
        c.block_table = _ptr(self.block_table)
        c.k_tensor_scale = _ptr(self.k_tensor_scale)
        c.v_tensor_scale = _ptr(self.v_tensor_scale)
        return c

    def seq_struct(self, b: int) -> LayerCache:
        """The cache struct of sequence b alone (pointer offsets), for batch = 1 calls."""
        c = self.struct()
        for n in FIELDS:
            if n != "block_pool" and getattr(c, n):
                setattr(c, n, getattr(c, n) + b * (self.sizes[n] // self.num_seqs))
        if self.block_table is not None:
            c.block_table = c.block_table + b * self.cfg.max_blocks_per_seq * 4
        return c

    def nbytes(self) -> int:
        return sum(self.sizes.values())

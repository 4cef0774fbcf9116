"""Seeded synthetic inputs for the quantized KV-cache decode path.

This module is shared by the tests, the benchmark and the oracle-side checks.
It holds no arithmetic of the quantization method itself: it only draws
normal samples, scales chosen "outlier" channels, rounds to bf16 (that is how
the inputs are defined) and describes the workload shapes.

Recipe (all seeded with numpy ``Generator(PCG64)``):

* every K, V and Q element is a standard normal sample, rounded to bf16 with
  round-to-nearest-even;
* a seeded set of outlier channels is multiplied by a fixed factor *before*
  the rounding (the pages' point that Keys carry a few large fixed channels:
  "KV Cache Quantization Analysis", section 3, "Key=per-channel,
  Value=per-token");
* sequence lengths for the paged workload are log-uniform, block tables are a
  seeded permutation of the block pool.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

# --------------------------------------------------------------------------- #
# bf16 helpers (input definition, not method arithmetic)
# --------------------------------------------------------------------------- #


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    rounded = u + np.uint32(0x7FFF) + lsb
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- #
# Workload descriptions
# --------------------------------------------------------------------------- #

FORMAT_BITS = {"int2": 2, "int4": 4, "int8": 8, "fp8_e4m3": 8, "fp8_e5m2": 8, "bf16": 16}


@dataclasses.dataclass(frozen=True)
class LayerFormat:
    """Quantization layout of one layer's KV cache.

    fmt: "int2" | "int4" | "int8" | "fp8_e4m3" | "fp8_e5m2" | "bf16" (a skip layer: nothing quantized)
    G:   Key group length in tokens (per-channel Key quantization); 1 for FP8
    Gv:  Value group width in channels (per-token Value quantization)
    R:   residual window: the most recent tokens kept in bf16
    S:   sink tokens kept in bf16 at the start of the sequence
    rope_base: > 0: Keys stored before RoPE and rotated at their position by the decode
    k_outliers, v_outliers: dense-and-sparse rows (entries per quantized row kept exactly)
    """

    fmt: str
    G: int
    Gv: int
    R: int
    S: int
    rope_base: float = 0.0
    k_outliers: int = 0
    v_outliers: int = 0


@dataclasses.dataclass
class Workload:
    name: str
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seq_len: Optional[int]            # uniform length (None when lengths are drawn)
    layer_formats: List[LayerFormat]  # one per layer
    k_outlier_channels: int           # per-head indices (count) or per-layer count, see outlier_mode
    v_outlier_channels: int
    outlier_scale: float
    outlier_mode: str                 # "per_head": same indices in every head; "per_layer": over Hkv*d
    paged: bool = False
    block_tokens: int = 16
    append_tokens: int = 0            # tokens appended by the timed decode step
    seq_len_range: Optional[Sequence[int]] = None  # (lo, hi) log-uniform, paged workload
    seed: int = 0
    n_query: int = 1                  # query tokens per sequence per step (the last n_query appended tokens)

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def tiny_int4() -> Workload:
    """Tiny KIVI INT4 decode: 1 layer, B=1, T=512, 8 q heads / 2 kv heads, d=128."""
    fmt = LayerFormat("int4", G=32, Gv=128, R=32, S=0)
    return Workload("tiny_kivi_int4", 1, 1, 8, 2, 128, 512, [fmt], 4, 0, 10.0, "per_head", seed=1001)


def llama3_8b_fp8() -> Workload:
    """Llama-3-8B-shaped decode layer, FP8 E4M3 KV with per-tensor fp32 scale."""
    fmt = LayerFormat("fp8_e4m3", G=1, Gv=128, R=0, S=0)
    return Workload("llama3_8b_fp8_e4m3", 1, 16, 32, 8, 128, 8192, [fmt], 10, 10, 8.0, "per_layer", seed=1002)


def llama3_8b_fp8_e5m2() -> Workload:
    """The same Llama-3-8B-shaped decode layer with FP8 E5M2 KV (the other OCP FP8 format)."""
    fmt = LayerFormat("fp8_e5m2", G=1, Gv=128, R=0, S=0)
    return Workload("llama3_8b_fp8_e5m2", 1, 16, 32, 8, 128, 8192, [fmt], 10, 10, 8.0, "per_layer", seed=1006)


def llama3_8b_bf16_skip() -> Workload:
    """The same layer left unquantized (a skip layer): bf16 K and V for every token, first token as sink."""
    fmt = LayerFormat("bf16", G=16, Gv=128, R=0, S=1)
    return Workload("llama3_8b_bf16_skip_layer", 1, 16, 32, 8, 128, 8192, [fmt], 10, 10, 8.0, "per_layer",
                    seed=1007)


def llama3_8b_fp8_2q() -> Workload:
    """The FP8 E4M3 8B layer verifying 2 speculative tokens per sequence: both are appended, and the
    2 x 4 query heads of each kv head attend causally in one launch."""
    fmt = LayerFormat("fp8_e4m3", G=1, Gv=128, R=0, S=0)
    return Workload("llama3_8b_fp8_e4m3_2q", 1, 16, 32, 8, 128, 8192, [fmt], 10, 10, 8.0, "per_layer",
                    append_tokens=2, seed=1008, n_query=2)


def llama3_8b_int4_prerope() -> Workload:
    """Llama-3-8B-shaped KIVI INT4 layer (B=16, T=8192, 32/8 heads, G=128, Gv=128, R=128) whose Keys are
    stored before RoPE (base 500000, Llama 3) and rotated at their positions by the decode."""
    fmt = LayerFormat("int4", G=128, Gv=128, R=128, S=0, rope_base=500000.0)
    return Workload("llama3_8b_kivi_int4_prerope", 1, 16, 32, 8, 128, 8192, [fmt], 4, 0, 10.0, "per_head",
                    seed=1009)


def llama3_8b_int4_sparse() -> Workload:
    """Llama-3-8B-shaped KIVI INT4 layer (B=16, T=8192, 32/8 heads, G=128, Gv=128, R=128) with dense-and-
    sparse rows: 2 Key and 2 Value entries of every quantized row (about 1.6 %) kept exactly."""
    fmt = LayerFormat("int4", G=128, Gv=128, R=128, S=0, k_outliers=2, v_outliers=2)
    return Workload("llama3_8b_kivi_int4_sparse", 1, 16, 32, 8, 128, 8192, [fmt], 4, 0, 10.0, "per_head",
                    seed=1010)


def llama3_70b_int4() -> Workload:
    """Llama-3-70B-shaped decode over 80 layers, KIVI INT4 (G=128, Gv=128, R=128)."""
    fmt = LayerFormat("int4", G=128, Gv=128, R=128, S=0)
    return Workload("llama3_70b_kivi_int4_80l", 80, 16, 64, 8, 128, 8192, [fmt] * 80, 4, 0, 10.0, "per_head",
                    seed=1003)


def llama2_7b_int2() -> Workload:
    """KIVI-2 INT2 long context, Llama-2-7B shape (MHA), one appended token per sequence."""
    fmt = LayerFormat("int2", G=32, Gv=32, R=128, S=0)
    return Workload("llama2_7b_kivi2_int2_32k", 1, 32, 32, 32, 128, 32768, [fmt], 3, 0, 12.0, "per_head",
                    append_tokens=1, seed=1004)


def paged_mixed() -> Workload:
    """Paged mixed-precision batch: 64 layers, INT8 on the first/last 4 layers, INT4 elsewhere."""
    int8 = LayerFormat("int8", G=16, Gv=128, R=64, S=1)
    int4 = LayerFormat("int4", G=16, Gv=128, R=64, S=1)
    fmts = [int8 if (l < 4 or l >= 60) else int4 for l in range(64)]
    return Workload("paged_mixed_int8_int4_64l", 64, 64, 48, 8, 128, None, fmts, 20, 0, 10.0, "per_layer",
                    paged=True, block_tokens=16, append_tokens=1, seq_len_range=(1024, 65536), seed=1005)


WORKLOADS = {
    "tiny_kivi_int4": tiny_int4,
    "llama3_8b_fp8_e4m3": llama3_8b_fp8,
    "llama3_8b_fp8_e5m2": llama3_8b_fp8_e5m2,
    "llama3_8b_bf16_skip_layer": llama3_8b_bf16_skip,
    "llama3_8b_fp8_e4m3_2q": llama3_8b_fp8_2q,
    "llama3_8b_kivi_int4_prerope": llama3_8b_int4_prerope,
    "llama3_8b_kivi_int4_sparse": llama3_8b_int4_sparse,
    "llama3_70b_kivi_int4_80l": llama3_70b_int4,
    "llama2_7b_kivi2_int2_32k": llama2_7b_int2,
    "paged_mixed_int8_int4_64l": paged_mixed,
}


# --------------------------------------------------------------------------- #
# Seeded draws
# --------------------------------------------------------------------------- #


def _stream(seed: int, name: str) -> np.random.Generator:
    # a named sub-stream: hash the name into the spawn key so streams are independent
    key = [int.from_bytes(name.encode(), "little") % (2 ** 32)]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=key)))


def outlier_channels(w: Workload, which: str, layer: int = 0) -> np.ndarray:
    """Boolean mask [Hkv, d] of channels multiplied by ``w.outlier_scale``.

    per_head: the same ``count`` indices (out of d) in every head and layer.
    per_layer: ``count`` indices drawn over the layer's Hkv*d channels.
    """
    count = w.k_outlier_channels if which == "k" else w.v_outlier_channels
    mask = np.zeros((w.num_kv_heads, w.head_dim), dtype=bool)
    if count == 0:
        return mask
    if w.outlier_mode == "per_head":
        rng = _stream(w.seed, f"outlier-{which}")
        idx = rng.choice(w.head_dim, size=count, replace=False)
        mask[:, idx] = True
    else:
        rng = _stream(w.seed, f"outlier-{which}-layer{layer}")
        idx = rng.choice(w.num_kv_heads * w.head_dim, size=count, replace=False)
        mask.reshape(-1)[idx] = True
    return mask


def seq_lens(w: Workload) -> np.ndarray:
    """Per-sequence lengths (tokens already in the cache before the timed step)."""
    if w.seq_len_range is None:
        return np.full(w.batch, w.seq_len - w.append_tokens, dtype=np.int64)
    lo, hi = w.seq_len_range
    rng = _stream(w.seed, "lengths")
    u = rng.random(w.batch)
    lens = np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))
    return np.floor(lens).astype(np.int64)


def kv_bf16(w: Workload, layer: int, b: int, h: int, T: int) -> (np.ndarray, np.ndarray):
    """K and V of one (layer, sequence, kv head): bf16 bits [T, d] each.

    Drawn from a stream keyed by (layer, b, h) so that any subset of heads can be
    regenerated on its own.
    """
    rng = _stream(w.seed, f"kv-l{layer}-b{b}-h{h}")
    k = rng.standard_normal((T, w.head_dim), dtype=np.float32)
    v = rng.standard_normal((T, w.head_dim), dtype=np.float32)
    km = outlier_channels(w, "k", layer)[h]
    vm = outlier_channels(w, "v", layer)[h]
    k[:, km] *= np.float32(w.outlier_scale)
    v[:, vm] *= np.float32(w.outlier_scale)
    return f32_to_bf16_bits(k), f32_to_bf16_bits(v)


def q_bf16(w: Workload, layer: int) -> np.ndarray:
    """Decode queries of one layer: bf16 bits [B, Hq, d]."""
    rng = _stream(w.seed, f"q-l{layer}")
    shape = (w.batch, w.num_q_heads, w.head_dim) if w.n_query == 1 else (w.batch, w.n_query, w.num_q_heads, w.head_dim)
    q = rng.standard_normal(shape, dtype=np.float32)
    return f32_to_bf16_bits(q)


def block_permutation(w: Workload, num_blocks: int, layer: int = 0) -> np.ndarray:
    """Seeded permutation of the block pool used to build block tables."""
    rng = _stream(w.seed, f"blocks-l{layer}")
    return rng.permutation(num_blocks).astype(np.int32)


def random_bf16(seed: int, shape, scale: float = 1.0, outlier_mask: Optional[np.ndarray] = None,
                outlier_scale: float = 1.0) -> np.ndarray:
    """Generic seeded N(0, scale^2) bf16 bits; ``outlier_mask`` broadcasts over the last axis."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal(shape, dtype=np.float32) * np.float32(scale)
    if outlier_mask is not None:
        x = np.where(outlier_mask, x * np.float32(outlier_scale), x).astype(np.float32)
    return f32_to_bf16_bits(x)


# --------------------------------------------------------------------------- #
# Device-side draws for full-size workloads (timing; sampled parity)
# --------------------------------------------------------------------------- #


def device_kv_bf16(w: Workload, layer: int, T: int, device, batch: Optional[int] = None, seed_offset: int = 0):
    """K, V of one layer for all sequences and kv heads: torch bf16 [B, H, T, d] on ``device``.

    Seeded torch generator on the device; outlier channels as in ``outlier_channels``.
    The bf16 values are the inputs: tests copy sampled (sequence, head) slices back to
    the host for the oracle.
    """
    import torch
    B = w.batch if batch is None else batch
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 100003 + layer * 7919 + seed_offset)
    shape = (B, w.num_kv_heads, T, w.head_dim)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    km = torch.from_numpy(outlier_channels(w, "k", layer)).to(device)
    vm = torch.from_numpy(outlier_channels(w, "v", layer)).to(device)
    scale = float(w.outlier_scale)
    k = torch.where(km[None, :, None, :], k * scale, k)
    v = torch.where(vm[None, :, None, :], v * scale, v)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def device_q_bf16(w: Workload, layer: int, device, batch: Optional[int] = None, seed_offset: int = 0):
    """Decode queries of one layer: torch bf16 [B, Hq, d] (or [B, n_query, Hq, d]) on ``device`` (seeded)."""
    import torch
    B = w.batch if batch is None else batch
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed * 100019 + layer * 104729 + seed_offset + 1)
    shape = (B, w.num_q_heads, w.head_dim) if w.n_query == 1 else (B, w.n_query, w.num_q_heads, w.head_dim)
    q = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return q.to(torch.bfloat16)

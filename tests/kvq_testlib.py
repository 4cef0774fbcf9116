"""Test helpers: drive libkvq through its C ABI and read its buffers back.

The physical-layout decoder below restates the layout contract written in
include/kvq.h (it is test code, independent of the CUDA sources); the oracle
side is oracle/kvq_oracle.py.  No expected value here comes from the GPU.
"""
from __future__ import annotations

import ctypes
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

from oracle import kvq_oracle as O

F32 = np.float32
BITS = {"int2": 2, "int4": 4, "int8": 8, "fp8_e4m3": 8, "fp8_e5m2": 8}


# --------------------------------------------------------------------------- #
# layout contract (include/kvq.h), restated for reading buffers back
# --------------------------------------------------------------------------- #


def _frag_positions(fmt: str, i: np.ndarray, k: np.ndarray, s: np.ndarray):
    """(byte, bit) of A-operand element (row i, column k) of step s (the header's fragment order)."""
    lane = 4 * (i % 8) + (k % 8) // 2
    reg = i // 8 + 2 * (k // 8)
    h = k % 2
    if fmt == "int4":
        w, bit = s, 4 * reg + 16 * h
    elif fmt == "int2":
        w, bit = s // 2, 8 * (s % 2) + 2 * reg + 16 * h
    elif fmt == "int8":
        w, bit = 2 * s + reg // 2, 8 * ((reg % 2) + 2 * h)
    else:  # fp8_e4m3, fp8_e5m2
        w, bit = 2 * s + reg // 2, 8 * (2 * (reg % 2) + h)
    byte = ((w // 4) * 32 + lane) * 16 + (w % 4) * 4 + bit // 8
    return byte, bit % 8


def ktile_positions(fmt: str):
    """(byte[16,128], bit[16,128]) of Key code (token, channel) in a tile's K part."""
    t = np.arange(16)[:, None] + 0 * np.arange(128)[None, :]
    c = 0 * np.arange(16)[:, None] + np.arange(128)[None, :]
    e = c % 4
    return _frag_positions(fmt, t, 2 * ((c // 4) % 4) + e % 2 + 8 * (e // 2), c // 16)


def vtile_positions(fmt: str):
    """(byte[16,128], bit[16,128]) of Value code (token, channel) in a tile's V part."""
    t = np.arange(16)[:, None] + 0 * np.arange(128)[None, :]
    c = 0 * np.arange(16)[:, None] + np.arange(128)[None, :]
    return _frag_positions(fmt, c % 16, t, c // 16)


def unpack_tiles(raw: np.ndarray, fmt: str, positions) -> np.ndarray:
    """Code matrices of tiles [ntiles, 16*rb] bytes -> codes [ntiles*16, 128]."""
    b = BITS[fmt]
    byte, bit = positions(fmt)
    raw = raw.astype(np.uint32)
    vals = (raw[:, byte] >> bit[None]) & ((1 << b) - 1)   # [ntiles, 16, 128]
    return vals.reshape(-1, 128).astype(np.uint8)


def bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x_f32, dtype=np.float32).view(np.uint32) >> 16


# --------------------------------------------------------------------------- #
# a GPU cache built through kvq_quantize_append
# --------------------------------------------------------------------------- #


class GpuLayer:
    """One layer's cache on the GPU for B sequences, with its oracle twin."""

    def __init__(self, fmt: str, H: int, lens: Sequence[int], G: int, Gv: int, R: int, S: int, *,
                 paged: bool = False, block_tokens: int = 16, spare_blocks: int = 3, seed: int = 0,
                 extra_capacity: int = 0, device="cuda", rope_base: float = 0.0, k_outliers: int = 0,
                 v_outliers: int = 0):
        import torch
        from quantized_kv_cache_decode_gb300 import kvq
        self.torch, self.kvq = torch, kvq
        self.fmt, self.H, self.lens = fmt, H, list(lens)
        self.B = len(lens)
        self.fp8 = fmt in ("fp8_e4m3", "fp8_e5m2")
        self.bf16 = fmt == "bf16"
        self.G = 1 if self.fp8 else (16 if self.bf16 else G)
        self.Gv = 128 if (self.fp8 or self.bf16) else Gv
        self.R = 0 if (self.fp8 or self.bf16) else R
        self.S = S
        self.spec = O.Spec(fmt, d=128, G=self.G, Gv=self.Gv, R=self.R, S=S, rope_base=rope_base,
                           k_outliers=k_outliers, v_outliers=v_outliers)
        self.nk, self.nv = k_outliers, v_outliers
        out_kw = dict(rope_base=rope_base, k_outliers=k_outliers, v_outliers=v_outliers)
        self.device = device
        self.paged = paged
        maxq = max([O.token_split(T + extra_capacity, self.spec)[1] for T in self.lens] + [0])
        unit = 16 if self.fp8 else max(16, self.G)
        if self.bf16:
            # every token after the sink in the bf16 buffers, row t - S
            self.W = max([1] + [T + extra_capacity - min(T + extra_capacity, S) for T in self.lens])
            self.cfg = kvq.make_config(fmt, H, 0, 0, 0, S, capacity_tokens=self.W)
        elif paged:
            self.P = block_tokens if self.fp8 else self.G
            blocks_per_seq = [math.ceil(O.token_split(T + extra_capacity, self.spec)[1] / self.P) for T in self.lens]
            self.mbps = max(blocks_per_seq + [1])
            nblocks = sum(blocks_per_seq) + spare_blocks
            self.cfg = kvq.make_config(fmt, H, self.G, self.Gv, self.R, S, paged=True, block_tokens=self.P,
                                       num_blocks=nblocks, max_blocks_per_seq=self.mbps, **out_kw)
        else:
            cap = max(unit, math.ceil(maxq / unit) * unit)
            self.cfg = kvq.make_config(fmt, H, self.G, self.Gv, self.R, S, capacity_tokens=cap, **out_kw)
        self.layer = kvq.CacheLayer(self.cfg, self.B, device=device)
        if paged:
            rng = np.random.default_rng(seed + 77)
            perm = rng.permutation(nblocks).astype(np.int32)
            table = np.full((self.B, self.mbps), -1, np.int32)
            k = 0
            for b, nb in enumerate(blocks_per_seq):
                table[b, :nb] = perm[k:k + nb]
                k += nb
            self.table_np = table
            self.layer.block_table.copy_(torch.from_numpy(table))
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    # -- per-sequence view of the cache struct (batch = 1 calls) --
    def seq_struct(self, b: int):
        return self.layer.seq_struct(b)

    def calibrate_fp8(self, k_all_bits: np.ndarray, v_all_bits: np.ndarray):
        torch = self.torch
        kd = torch.from_numpy(k_all_bits.astype(np.int16)).to(self.device)
        vd = torch.from_numpy(v_all_bits.astype(np.int16)).to(self.device)
        self.kvq.fp8_calibrate(kd, kd.numel(), self.layer.k_tensor_scale, fmt=self.fmt)
        self.kvq.fp8_calibrate(vd, vd.numel(), self.layer.v_tensor_scale, fmt=self.fmt)
        torch.cuda.synchronize()

    def append(self, b: int, k_bits: np.ndarray, v_bits: np.ndarray, T_before: int):
        """Append tokens [n, d] (bf16 bits) to every kv head of sequence b (k_bits: [H, n, d])."""
        torch = self.torch
        n = k_bits.shape[1]
        kd = torch.from_numpy(np.ascontiguousarray(k_bits).astype(np.int16)).to(self.device)
        vd = torch.from_numpy(np.ascontiguousarray(v_bits).astype(np.int16)).to(self.device)
        sl = torch.tensor([T_before], dtype=torch.int32, device=self.device)
        self.kvq.quantize_append(self.cfg, self.seq_struct(b), kd, vd, n, sl, 1, self.status)

    def seq_lens_dev(self, lens=None):
        return self.torch.tensor(self.lens if lens is None else lens, dtype=self.torch.int32, device=self.device)

    def raw(self, name: str) -> np.ndarray:
        return self.layer.buf[name].cpu().numpy()

    def status_value(self) -> int:
        return int(self.status.item())

    def decode(self, q_bits: np.ndarray, out_bf16: bool = False, lens=None, scale=None):
        torch = self.torch
        B, Hq, _ = q_bits.shape
        qd = torch.from_numpy(q_bits.astype(np.int16)).to(self.device)
        out = torch.zeros((B, Hq, 128), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=self.device)
        lse = torch.zeros((B, Hq), dtype=torch.float32, device=self.device)
        wsb = self.kvq.decode_workspace_size(self.cfg, B, Hq)
        ws = torch.zeros(wsb, dtype=torch.uint8, device=self.device)
        sl = self.seq_lens_dev(lens)
        sc = 1.0 / math.sqrt(128) if scale is None else scale
        self.kvq.decode_attention(self.cfg, self.layer.struct(), qd, Hq, sl, B, sc, out, out_bf16, lse, ws, wsb,
                                  self.status)
        torch.cuda.synchronize()
        return out, lse

    def append_decode(self, k_bits: np.ndarray, v_bits: np.ndarray, q_bits: np.ndarray, lens_before,
                      out_bf16: bool = False):
        """One whole step (kvq_append_decode_attention): k_bits, v_bits [B, H, d] the step's token."""
        torch = self.torch
        B, Hq, _ = q_bits.shape
        qd = torch.from_numpy(q_bits.astype(np.int16)).to(self.device)
        kd = torch.from_numpy(np.ascontiguousarray(k_bits).astype(np.int16)).to(self.device)
        vd = torch.from_numpy(np.ascontiguousarray(v_bits).astype(np.int16)).to(self.device)
        out = torch.zeros((B, Hq, 128), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=self.device)
        lse = torch.zeros((B, Hq), dtype=torch.float32, device=self.device)
        wsb = self.kvq.decode_workspace_size(self.cfg, B, Hq)
        ws = torch.zeros(wsb, dtype=torch.uint8, device=self.device)
        self.kvq.append_decode_attention(self.cfg, self.layer.struct(), kd, vd, self.seq_lens_dev(lens_before), B, qd,
                                         Hq, 1.0 / math.sqrt(128), out, out_bf16, lse, ws, wsb, self.status)
        torch.cuda.synchronize()
        return out, lse

    def decode_multi(self, q_bits: np.ndarray, out_bf16: bool = False, scale=None):
        """q_bits [B, M, Hq, d]: the last M cached tokens' queries, attending causally."""
        torch = self.torch
        B, M, Hq, _ = q_bits.shape
        qd = torch.from_numpy(np.ascontiguousarray(q_bits).astype(np.int16)).to(self.device)
        out = torch.zeros((B, M, Hq, 128), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=self.device)
        lse = torch.zeros((B, M, Hq), dtype=torch.float32, device=self.device)
        wsb = self.kvq.decode_workspace_size_multi(self.cfg, B, M, Hq)
        ws = torch.zeros(wsb, dtype=torch.uint8, device=self.device)
        sc = 1.0 / math.sqrt(128) if scale is None else scale
        self.kvq.decode_attention_multi(self.cfg, self.layer.struct(), qd, M, Hq, self.seq_lens_dev(), B, sc, out,
                                        out_bf16, lse, ws, wsb, self.status)
        torch.cuda.synchronize()
        return out, lse

    def dequantize(self, max_tokens: int, lens=None):
        torch = self.torch
        ko = torch.full((self.B, self.H, max_tokens, 128), 7.0, dtype=torch.float32, device=self.device)
        vo = torch.full_like(ko, 7.0)
        self.kvq.dequantize(self.cfg, self.layer.struct(), self.seq_lens_dev(lens), self.B, max_tokens, ko, vo,
                            self.status)
        torch.cuda.synchronize()
        return ko.cpu().numpy(), vo.cpu().numpy()

    # -- read the stored cache of (b, h) back into the oracle's logical form --
    def _layout(self):
        rb = 128 * BITS.get(self.fmt, 8) // 8
        ngv = 128 // self.Gv
        tile = 32 * rb + (0 if self.fp8 else 128 * ngv + 64 * (self.nk + self.nv))
        hdr = 0 if self.fp8 else 1024
        tpg = (self.P // 16) if self.paged else (1 if self.fp8 else self.G // 16)
        return rb, ngv, tile, hdr, tpg, hdr + tpg * tile

    def _record(self, b: int, h: int, ri: int) -> np.ndarray:
        rb, ngv, tile, hdr, tpg, rec = self._layout()
        if self.paged:
            pool = self.raw("block_pool")
            blk = int(self.table_np[b, ri])
            base = blk * rec * self.H + h * rec
            return pool[base:base + rec]
        store = self.raw("qstore")
        nrec = self.cfg.capacity_tokens // (16 * tpg)
        base = ((b * self.H + h) * nrec + ri) * rec
        return store[base:base + rec]

    def logical(self, b: int, h: int, T: int) -> Dict[str, np.ndarray]:
        n_sink, qn, r = O.token_split(T, self.spec)
        rb, ngv, tile, hdr, tpg, rec = self._layout()
        kc, vt, ks, kz, vs, vz, kspl, vspl = [], [], [], [], [], [], [], []
        ntiles = (qn + 15) // 16
        for i in range(ntiles):
            recb = self._record(b, h, i // tpg)
            t = recb[hdr + (i % tpg) * tile: hdr + (i % tpg + 1) * tile]
            kc.append(t[:16 * rb].reshape(1, 16 * rb))
            vt.append(t[16 * rb:32 * rb].reshape(1, 16 * rb))
            if not self.fp8:
                vs.append(t[32 * rb:32 * rb + 64 * ngv].view(F32).reshape(16, ngv))
                vz.append(t[32 * rb + 64 * ngv:32 * rb + 128 * ngv].view(F32).reshape(16, ngv))
                sp0 = 32 * rb + 128 * ngv
                kspl.append(t[sp0:sp0 + 64 * self.nk].view(np.uint32).reshape(16, self.nk))
                vspl.append(t[sp0 + 64 * self.nk:sp0 + 64 * (self.nk + self.nv)].view(np.uint32).reshape(16, self.nv))
                if i % tpg == 0:
                    ks.append(recb[:512].view(F32).reshape(1, 128))
                    kz.append(recb[512:1024].view(F32).reshape(1, 128))
        out = {}
        kc = np.concatenate(kc) if kc else np.zeros((0, 16 * rb), np.uint8)
        vt = np.concatenate(vt) if vt else np.zeros((0, 16 * rb), np.uint8)
        if not self.fp8:
            out["k_s"] = np.concatenate(ks)[:qn // self.G] if ks else np.zeros((0, 128), F32)
            out["k_z"] = np.concatenate(kz)[:qn // self.G] if kz else np.zeros((0, 128), F32)
            out["v_s"] = np.concatenate(vs)[:qn] if vs else np.zeros((0, ngv), F32)
            out["v_z"] = np.concatenate(vz)[:qn] if vz else np.zeros((0, ngv), F32)
            # dense-and-sparse entries: bf16 bits << 16 | channel
            ke = np.concatenate(kspl)[:qn] if kspl else np.zeros((0, self.nk), np.uint32)
            ve = np.concatenate(vspl)[:qn] if vspl else np.zeros((0, self.nv), np.uint32)
            out["k_sp_idx"], out["k_sp_bits"] = (ke & 127).astype(np.int64), (ke >> 16).astype(np.uint16)
            out["v_sp_idx"], out["v_sp_bits"] = (ve & 127).astype(np.int64), (ve >> 16).astype(np.uint16)
        out["k_codes"] = unpack_tiles(kc, self.fmt, ktile_positions)[:qn] if len(kc) else np.zeros((0, 128), np.uint8)
        out["v_codes"] = unpack_tiles(vt, self.fmt, vtile_positions)[:qn] if len(vt) else np.zeros((0, 128), np.uint8)
        pair = b * self.H + h
        if n_sink:
            sk = self.raw("sink_k").view(np.uint16).reshape(self.B * self.H, self.S, 128)[pair, :n_sink]
            sv = self.raw("sink_v").view(np.uint16).reshape(self.B * self.H, self.S, 128)[pair, :n_sink]
            out["sink_k"], out["sink_v"] = sk, sv
        if not self.fp8:
            W = self.W if self.bf16 else self.R + self.G
            ring_k = self.raw("resid_k").view(np.uint16).reshape(self.B * self.H, W, 128)[pair]
            ring_v = self.raw("resid_v").view(np.uint16).reshape(self.B * self.H, W, 128)[pair]
            slots = [(qn + i) % W for i in range(r)]
            out["resid_k"], out["resid_v"] = ring_k[slots], ring_v[slots]
        return out


def compare_logical(gpu: Dict[str, np.ndarray], hc: "O.HeadCache"):
    """Bit-exact comparison of a GPU head cache (logical form) with the oracle's."""
    assert np.array_equal(gpu["k_codes"], hc.k_codes), "K codes differ"
    assert np.array_equal(gpu["v_codes"], hc.v_codes), "V codes differ"
    if hc.k_s is not None:
        for f in ("k_s", "k_z", "v_s", "v_z"):
            g, o = gpu[f], getattr(hc, f)
            assert g.shape == o.shape and np.array_equal(g.view(np.uint32), o.astype(F32).view(np.uint32)), f
        for kv in ("k", "v"):  # dense-and-sparse lists
            assert np.array_equal(gpu[kv + "_sp_idx"], getattr(hc, kv + "_sp_idx")), kv + " sparse channels"
            assert np.array_equal(gpu[kv + "_sp_bits"], bf16_bits(getattr(hc, kv + "_sp_val"))), kv + " sparse values"
    if len(hc.sink_k):
        assert np.array_equal(gpu["sink_k"], bf16_bits(hc.sink_k)) and np.array_equal(gpu["sink_v"], bf16_bits(hc.sink_v))
    if not hc.spec.is_fp8:
        assert np.array_equal(gpu["resid_k"], bf16_bits(hc.resid_k)), "residual K differs"
        assert np.array_equal(gpu["resid_v"], bf16_bits(hc.resid_v)), "residual V differs"


def check_attention(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray, lse_ref: np.ndarray,
                    rel: float = 2e-3, lse_tol: float = 1e-4):
    """The parity bar: max|out - ref| <= rel * max|ref| over the tensor; |lse - ref| <= lse_tol."""
    finite = np.isfinite(lse_ref)
    scale = np.max(np.abs(out_ref)) if out_ref.size else 0.0
    err = np.max(np.abs(out_gpu.astype(np.float64) - out_ref)) if out_ref.size else 0.0
    assert err <= rel * scale + 1e-30, f"max |out err| {err:.3e} > {rel} * {scale:.3e}"
    if finite.any():
        lerr = np.max(np.abs(lse_gpu.astype(np.float64)[finite] - lse_ref[finite]))
        assert lerr <= lse_tol, f"max |lse err| {lerr:.3e} > {lse_tol}"
    assert np.all(np.isneginf(lse_gpu[~finite])), "empty sequences must give lse = -inf"
    return err / scale if scale else 0.0, (np.max(np.abs(lse_gpu[finite] - lse_ref[finite])) if finite.any() else 0.0)

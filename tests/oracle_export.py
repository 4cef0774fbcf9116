"""Oracle side of the all-pairs export check, run in spawned worker processes.

Imports numpy and the oracle only, so a worker starts quickly and never touches
the GPU.  A worker rebuilds one (sequence, kv head) cache from its bf16 inputs,
the way the benchmark step builds it (the first T - n_app tokens in one append,
then the step's n_app tokens one at a time), and returns the sha256 of the
dequantized export's fp32 bit patterns for K and for V.
"""
import hashlib

import numpy as np

from oracle import kvq_oracle as O


def digest(x: np.ndarray) -> str:
    """sha256 of an fp32 array's bit patterns (C order)."""
    a = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return hashlib.sha256(memoryview(a).cast("B")).hexdigest()


def export_digests(spec, k_bits: np.ndarray, v_bits: np.ndarray, n_app: int, k_scale=None, v_scale=None):
    """(digest of K's export, digest of V's export) for K, V given as bf16 bits [T, d]."""
    k = O.bf16_to_f32(k_bits)
    v = O.bf16_to_f32(v_bits)
    T = len(k)
    hc = O.build_head_cache(k[:T - n_app], v[:T - n_app], spec, k_scale, v_scale)
    for t in range(T - n_app, T):
        O.append_token(hc, k[t], v[t])
    kr, vr = O.dequantized_f32(hc)
    return digest(kr), digest(vr)

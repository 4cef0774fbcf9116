"""The roofline numerator: bench.py's algorithmic byte counts against closed forms.

Each expected value is written out from the cache layout's definition (codes at b
bits per element for K and V, fp32 scale + zero-point per Key group channel and per
Value token group, bf16 K and V for sink and residual tokens, bf16 q and out and an
fp32 lse per query row; the KV part is the box "메모리 크기 감각" of "KV Cache
Quantization Analysis" with the per-group metadata added), independently of the
accounting functions in bench.py.
"""
import numpy as np

import bench
from quantized_kv_cache_decode_gb300 import inputs as I


def _qol(rows):  # q and out in bf16, lse in fp32
    return rows * (128 * 2 * 2 + 4)


def _attention(w, T):
    return sum(bench.attention_bytes(f, T, w.num_kv_heads) for f in w.layer_formats[:1]) * w.batch


def test_tiny_int4():
    w = I.tiny_int4()  # B=1, H=2, Hq=8, T=512, INT4, G=32, Gv=128, R=32 -> Q_n = 480, r = 32
    pairs = 1 * 2
    codes = pairs * 2 * 480 * 128 // 2
    k_sz = pairs * (480 // 32) * 128 * 8
    v_sz = pairs * 480 * 1 * 8
    resid = pairs * 32 * 128 * 2 * 2
    assert (codes, k_sz, v_sz, resid) == (122880, 30720, 7680, 32768)
    assert _attention(w, 512) + _qol(8) == 198176 == codes + k_sz + v_sz + resid + _qol(8)


def test_llama3_8b_fp8_step():
    w = I.llama3_8b_fp8()  # B=16, H=8, Hq=32, T=8192, FP8: one byte per element, no metadata
    pairs = 16 * 8
    attn = pairs * 2 * 8192 * 128 + _qol(16 * 32)
    assert _attention(w, 8192) + _qol(16 * 32) == attn == 268699648
    # the step also appends one token per pair: read the new K, V (bf16), write their codes
    app = pairs * (2 * 128 * 2 + 2 * 128)
    assert bench.step_bytes(w, np.full(16, 8192), 1) == attn + app == 268797952


def test_llama3_70b_int4_layer():
    w = I.llama3_70b_int4()  # B=16, H=8, Hq=64, T=8192, INT4 G=128 Gv=128 R=128 -> Q_n = 8064, r = 128
    pairs = 16 * 8
    codes = pairs * 2 * 8064 * 128 // 2
    k_sz = pairs * (8064 // 128) * 128 * 8
    v_sz = pairs * 8064 * 1 * 8
    resid = pairs * 128 * 128 * 2 * 2
    per_layer = codes + k_sz + v_sz + resid + _qol(16 * 64)
    assert per_layer == 157552640
    assert _attention(w, 8192) + _qol(16 * 64) == per_layer
    assert 80 * per_layer == 12604211200  # the 80-layer step, about 12.6 GB


def test_llama2_7b_int2_step_with_spill():
    w = I.llama2_7b_int2()  # B=32, H=Hq=32, INT2 G=32 Gv=32 R=128; 32767 tokens, +1 -> 32768
    pairs = 32 * 32
    qn, r = 32640, 128  # after the append the window (160 = R + G tokens) spilled one group
    codes = pairs * 2 * qn * 128 // 4
    k_sz = pairs * (qn // 32) * 128 * 8
    v_sz = pairs * qn * 4 * 8
    resid = pairs * r * 128 * 2 * 2
    attn = codes + k_sz + v_sz + resid + _qol(32 * 32)
    # append: read the new K, V; write them to the ring; read back the 32 spilled tokens
    # (bf16 K, V); write their codes, the group's K scale/zero and the tokens' V scale/zero
    app = pairs * (512 + 512 + 32 * 128 * 2 * 2 + 2 * 32 * 128 // 4 + 128 * 8 + 32 * 4 * 8)
    assert app == 22020096
    assert bench.step_bytes(w, np.full(32, 32768), 1) == attn + app == 4367847424


def test_launch_count_claim():
    # the bench's gpu_launches: append + decode per layer, one launch for FP8 layers without
    # sink tokens stepped through kvq_append_decode_attention (one token, one query)
    assert bench.count_launches(I.llama3_8b_fp8()) == 1
    assert bench.count_launches(I.llama3_8b_fp8_e5m2()) == 1
    assert bench.count_launches(I.llama3_8b_fp8_2q()) == 2
    assert bench.count_launches(I.llama3_70b_int4()) == 160
    assert bench.count_launches(I.paged_mixed()) == 128

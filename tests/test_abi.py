"""The C-ABI library: it loads, exports every entry point include/kvq.h declares,
and its host-side validation and layout arithmetic work without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    import quantized_kv_cache_decode_gb300 as pkg
    pkg.build()
    from quantized_kv_cache_decode_gb300 import kvq as mod
    return mod


def test_exports_every_declared_symbol(kvq):
    declared = kvq.declared_symbols()
    assert set(declared) >= {"kvq_quantize_append", "kvq_decode_attention", "kvq_dequantize",
                             "kvq_cache_layout", "kvq_decode_workspace_size", "kvq_fp8_calibrate",
                             "kvq_status_string"}
    lib = ctypes.CDLL(kvq.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_binding_matches_declared_parameter_counts(kvq):
    # every entry point of include/kvq.h is bound with as many ctypes arguments as it declares
    with open(os.path.join(ROOT, "include", "kvq.h")) as f:
        text = f.read()
    decls = re.findall(r"^\s*(?:kvq_status|const char\*)\s+(kvq_\w+)\s*\(([^;]*?)\)\s*;", text, re.M | re.S)
    assert len(decls) == len(kvq.declared_symbols())
    for name, params in decls:
        n = len([p for p in params.split(",") if p.strip() and p.strip() != "void"])
        bound = getattr(kvq._lib, name).argtypes
        assert bound is not None and len(bound) == n, (name, n, bound)


def test_status_strings(kvq):
    for code, name in kvq.STATUS.items():
        assert kvq.status_string(code).startswith(name)


def test_cache_layout_sizes(kvq):
    # Llama-3-70B-shaped INT4 layer, contiguous: a record per 128-token Key group =
    # 1 KB header (fp32 K scale + zero) + 8 tiles of (2 x 1 KB codes + 16 x (4 + 4) B V scale/zero)
    cfg = kvq.make_config("int4", 8, 128, 128, 128, 0, capacity_tokens=8064)
    sz = kvq.cache_layout(cfg, 16)
    pairs = 16 * 8
    tile = 2 * 16 * 64 + 16 * 8
    assert sz["qstore"] == pairs * (8064 // 128) * (1024 + 8 * tile)
    assert sz["resid_k"] == pairs * 256 * 128 * 2 and sz["sink_k"] == 0 and sz["block_pool"] == 0
    # paged INT4, block 16 = G: one record per block and head = 1024 + 2048 + 128 = 3200 B
    cfg = kvq.make_config("int4", 8, 16, 128, 64, 1, paged=True, block_tokens=16, num_blocks=10,
                          max_blocks_per_seq=4)
    sz = kvq.cache_layout(cfg, 2)
    assert sz["block_pool"] == 10 * 8 * 3200
    assert sz["sink_k"] == 2 * 8 * 1 * 128 * 2
    # FP8: 1 B per element, no scales, no ring
    cfg = kvq.make_config("fp8_e4m3", 8, 1, 128, 0, 0, capacity_tokens=8192)
    sz = kvq.cache_layout(cfg, 16)
    assert sz["qstore"] == 16 * 8 * 8192 * 128 * 2 and sz["resid_k"] == 0
    cfg = kvq.make_config("fp8_e5m2", 8, 1, 128, 0, 0, capacity_tokens=8192)
    assert kvq.cache_layout(cfg, 16) == sz
    # bf16 skip layer: no quantized store, bf16 rows for every token after the sink
    cfg = kvq.make_config("bf16", 8, 0, 0, 0, 1, capacity_tokens=8191)
    sz = kvq.cache_layout(cfg, 16)
    assert sz["qstore"] == 0 and sz["block_pool"] == 0
    assert sz["resid_k"] == sz["resid_v"] == 16 * 8 * 8191 * 128 * 2
    assert sz["sink_k"] == 16 * 8 * 1 * 128 * 2


@pytest.mark.parametrize("kw,status", [
    (dict(fmt="int4", num_kv_heads=0, G=32, Gv=128, R=0, S=0, capacity_tokens=64), -1),
    (dict(fmt="int4", num_kv_heads=2, G=24, Gv=128, R=0, S=0, capacity_tokens=48), -1),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=48, R=0, S=0, capacity_tokens=64), -1),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=-1, S=0, capacity_tokens=64), -1),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=0, S=0, capacity_tokens=40), -1),
    (dict(fmt="fp8_e4m3", num_kv_heads=2, G=16, Gv=128, R=0, S=0, capacity_tokens=64), -1),
    (dict(fmt="fp8_e4m3", num_kv_heads=2, G=1, Gv=128, R=8, S=0, capacity_tokens=64), -1),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=0, S=0, paged=True, block_tokens=16, num_blocks=4,
          max_blocks_per_seq=2), -1),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=0, S=0, capacity_tokens=64, head_dim=64), -2),
    (dict(fmt="fp8_e5m2", num_kv_heads=2, G=16, Gv=128, R=0, S=0, capacity_tokens=64), -1),
    (dict(fmt="bf16", num_kv_heads=2, G=0, Gv=0, R=0, S=1, capacity_tokens=0), -1),
    (dict(fmt="bf16", num_kv_heads=2, G=0, Gv=0, R=0, S=0, paged=True, block_tokens=16, num_blocks=4,
          max_blocks_per_seq=2), -2),
    # Key groups longer than the append kernel stages in shared memory (256 tokens)
    (dict(fmt="int4", num_kv_heads=2, G=272, Gv=128, R=0, S=0, capacity_tokens=272), -2),
    # pre-RoPE Keys: integer formats with Value groups of 64 or 128 channels; a base above 1
    (dict(fmt="fp8_e4m3", num_kv_heads=2, G=1, Gv=128, R=0, S=0, capacity_tokens=64, rope_base=1e4), -2),
    (dict(fmt="bf16", num_kv_heads=2, G=0, Gv=0, R=0, S=1, capacity_tokens=64, rope_base=1e4), -2),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=32, R=0, S=0, capacity_tokens=64, rope_base=1e4), -2),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=0, S=0, capacity_tokens=64, rope_base=0.5), -1),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=0, S=0, capacity_tokens=64, rope_base=float("nan")), -1),
    # dense-and-sparse rows: 0..8 entries, integer formats, Gv of 64 or 128, not with pre-RoPE Keys
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=0, S=0, capacity_tokens=64, k_outliers=9), -1),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=0, S=0, capacity_tokens=64, v_outliers=-1), -1),
    (dict(fmt="fp8_e4m3", num_kv_heads=2, G=1, Gv=128, R=0, S=0, capacity_tokens=64, k_outliers=1), -2),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=16, R=0, S=0, capacity_tokens=64, v_outliers=1), -2),
    (dict(fmt="int4", num_kv_heads=2, G=32, Gv=128, R=0, S=0, capacity_tokens=64, k_outliers=1,
          rope_base=1e4), -2),
])
def test_config_validation(kvq, kw, status):
    kw = dict(kw)
    cfg = kvq.make_config(kw.pop("fmt"), kw.pop("num_kv_heads"), kw.pop("G"), kw.pop("Gv"), kw.pop("R"),
                          kw.pop("S"), **kw)
    with pytest.raises(kvq.KvqError) as e:
        kvq.cache_layout(cfg, 1)
    assert e.value.status == status


def test_calibrate_rejects_non_fp8_formats(kvq):
    with pytest.raises(kvq.KvqError) as e:
        kvq.fp8_calibrate(0, 0, 16, stream=0, fmt="int4")
    assert e.value.status == -1


def test_selftest_rejects_before_any_launch(kvq):
    cache = kvq.LayerCache()
    paged = kvq.make_config("int4", 2, 16, 128, 16, 0, paged=True, block_tokens=16, num_blocks=4, max_blocks_per_seq=2)
    with pytest.raises(kvq.KvqError) as e:
        kvq.selftest_bounded_wait(paged, cache, 0, 8, 0, 1, 0.1, 0, False, 0, 0, 0, 0, stream=0)
    assert e.value.status == -2
    cfg = kvq.make_config("fp8_e4m3", 2, 1, 128, 0, 0, capacity_tokens=64)
    with pytest.raises(kvq.KvqError) as e:  # no status word to report into
        kvq.selftest_bounded_wait(cfg, cache, 0, 8, 0, 1, 0.1, 16, False, 0, 0, 0, None, stream=0)
    assert e.value.status == -1


def test_lse_merge_rejects_bad_arguments(kvq):
    for args in ((16, 16, 0, 4, 16, 0), (16, 16, 2, 4, 16, 2), (0, 16, 2, 4, 16, 0), (16, 16, 2, 4, 8, 0)):
        o, l, n, rows, out, bf = args
        with pytest.raises(kvq.KvqError) as e:
            kvq.lse_merge(o, l, n, rows, out, bf, None, stream=0)
        assert e.value.status == -1


def test_calls_reject_bad_arguments_before_any_launch(kvq):
    cfg = kvq.make_config("int4", 2, 32, 128, 32, 0, capacity_tokens=64)
    cache = kvq.LayerCache()  # all NULL
    with pytest.raises(kvq.KvqError) as e:
        kvq.quantize_append(cfg, cache, 0, 0, 1, 0, 1, stream=0)
    assert e.value.status == -1
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attention(cfg, cache, 0, 8, 0, 1, 0.1, 0, False, 0, 0, 0, stream=0)
    assert e.value.status == -1
    with pytest.raises(kvq.KvqError) as e:
        kvq.dequantize(cfg, cache, 0, 1, 16, 0, 0, stream=0)
    assert e.value.status == -1


@pytest.mark.parametrize("part", ["k", "v"])
def test_fragment_order_is_a_bijection(part):
    # every bit of a tile's K (V) code matrix holds exactly one (token, channel) code
    import numpy as np
    import kvq_testlib as TL
    positions = TL.ktile_positions if part == "k" else TL.vtile_positions
    for fmt, bits in (("int2", 2), ("int4", 4), ("int8", 8), ("fp8_e4m3", 8), ("fp8_e5m2", 8)):
        byte, bit = positions(fmt)
        tile_bytes = 16 * 128 * bits // 8
        used = np.zeros(tile_bytes * 8, int)
        for t in range(16):
            for c in range(128):
                for k in range(bits):
                    used[byte[t, c] * 8 + bit[t, c] + k] += 1
        assert used.min() == 1 and used.max() == 1, fmt


def test_fragment_order_lane_words():
    # lane l's words are the 16-byte chunks l, l + 32, ... of the matrix: the K code of
    # (token t, channel c) and the V code of (token t, channel c) are held by the lanes
    # the tensor-core operand layout names (row t mod 8 / channel mod 8, column pair)
    import numpy as np
    import kvq_testlib as TL
    for fmt in ("int2", "int4", "int8", "fp8_e4m3"):
        kb, _ = TL.ktile_positions(fmt)
        vb, _ = TL.vtile_positions(fmt)
        t = np.arange(16)[:, None]
        c = np.arange(128)[None, :]
        assert np.array_equal((kb // 16) % 32, 4 * (t % 8) + (c // 4) % 4 + 0 * c)
        assert np.array_equal((vb // 16) % 32, 4 * (c % 8) + (t % 8) // 2)


def test_append_rejects_unaligned_inputs_before_any_launch(kvq):
    # the spill kernel stages new rows with 16-byte loads: k_new / v_new must be 16-byte aligned
    # (the cache pointers below are fake, aligned and never dereferenced: the call returns first)
    cfg = kvq.make_config("int4", 2, 32, 128, 32, 0, capacity_tokens=64)
    cache = kvq.LayerCache()
    cache.qstore, cache.resid_k, cache.resid_v = 1 << 20, 2 << 20, 3 << 20
    for kn, vn in ((4096 + 2, 8192), (4096, 8192 + 8)):
        with pytest.raises(kvq.KvqError) as e:
            kvq.quantize_append(cfg, cache, kn, vn, 1, 16, 1, stream=0)
        assert e.value.status == -1


def test_append_decode_host_errors_come_first(kvq):
    # kvq_append_decode_attention checks everything the host can before its first launch
    # (fake aligned pointers, never dereferenced)
    cfg = kvq.make_config("fp8_e4m3", 2, 1, 128, 0, 0, capacity_tokens=64)
    cache = kvq.LayerCache()
    cases = [dict(out_bf16=2), dict(k_new=4096 + 2), dict(v_new=0), dict(out=0)]
    for bad in cases:
        a = dict(k_new=4096, v_new=8192, out=12288, out_bf16=0)
        a.update(bad)
        with pytest.raises(kvq.KvqError) as e:
            kvq.append_decode_attention(cfg, cache, a["k_new"], a["v_new"], 16, 1, 32, 8, 0.1, a["out"],
                                        a["out_bf16"], 0, 0, 0, stream=0)
        assert e.value.status == -1, bad


def test_pre_rope_keys_reject_several_query_tokens(kvq):
    # the multi-query decode does not rotate Keys: refused before anything is enqueued
    cfg = kvq.make_config("int4", 2, 32, 128, 32, 0, capacity_tokens=64, rope_base=10000.0)
    cache = kvq.LayerCache()
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attention_multi(cfg, cache, 0, 2, 8, 0, 1, 0.1, 4096, False, 0, 0, 0, 0, stream=0)
    assert e.value.status == -2


def test_outlier_layout_sizes(kvq):
    # a dense-and-sparse tile carries 16 x (k + v) entries of 4 bytes after the Value scales
    cfg = kvq.make_config("int4", 8, 16, 128, 64, 1, paged=True, block_tokens=16, num_blocks=10,
                          max_blocks_per_seq=4, k_outliers=2, v_outliers=3)
    assert kvq.cache_layout(cfg, 2)["block_pool"] == 10 * 8 * (3200 + 64 * 5)

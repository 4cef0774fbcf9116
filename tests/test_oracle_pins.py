"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU.  Each test checks the oracle against something other than itself:
worked numbers printed on the pages (tests/golden/), closed forms, invariants of
the affine formula, and brute force on tiny inputs written here independently
(plain Python loops, ``math.exp``, exhaustive candidate search).
"""
import math

import numpy as np
import pytest

from conftest import read_golden
from oracle import kvq_oracle as O

F32 = np.float32


# --------------------------------------------------------------------------- #
# byte accounting: worked numbers on the pages
# --------------------------------------------------------------------------- #


def test_kv_size_closed_form_llama3_70b():
    g = read_golden("kv_size_llama3_70b.txt")
    args = (g["layers"], g["kv_heads"], g["head_dim"], g["seq_len"], g["batch"])
    bf16 = O.kv_cache_bytes(*args, 2)
    assert bf16 == g["bf16_bytes"]
    assert bf16 == g["bf16_gib"] * 2 ** 30
    assert O.kv_cache_bytes(*args, 1) == g["fp8_gib"] * 2 ** 30
    assert O.kv_cache_bytes(*args, 0.5) == g["int4_gib"] * 2 ** 30
    assert O.kv_cache_bytes(*args, 0.25) == g["int2_gib"] * 2 ** 30


def test_per_token_bytes_table():
    g = read_golden("per_token_kv_bytes.txt")
    # the fp8 row fixes the number of cached elements per token (1 byte each)
    elems = g["fp8_e4m3_kib"] * 1024
    q8 = O.block_format_bits_per_element(8, g["block"], g["scale_bits"])
    q4 = O.block_format_bits_per_element(4, g["block"], g["scale_bits"])
    assert q8 == 8.5 and q4 == 4.5
    assert elems * q8 / 8 == g["q8_0_kib"] * 1024
    assert elems * q4 / 8 == g["q4_0_kib"] * 1024
    ctx = g["context_tokens"]
    for kib, gib in ((g["q8_0_kib"], g["q8_0_gib_64k"]), (g["fp8_e4m3_kib"], g["fp8_e4m3_gib_64k"]),
                     (g["q4_0_kib"], g["q4_0_gib_64k"])):
        size = kib * 1024 * ctx / 2 ** 30
        assert abs(size - gib) <= 0.005 + 1e-12


# --------------------------------------------------------------------------- #
# affine quantizer
# --------------------------------------------------------------------------- #


def _groups(seed, shape, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(F32) * F32(scale)
    x[..., 0] += F32(3.0)   # off-centre groups (asymmetric case)
    return x


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_codes_in_range_and_endpoints(bits):
    x = _groups(bits, (300, 37), 5.0)
    q, s, z = O.affine_quantize(x, bits)
    assert q.dtype == np.uint8 and q.max() <= 2 ** bits - 1
    rows = np.arange(x.shape[0])
    assert np.all(q[rows, x.argmin(axis=1)] == 0)
    assert np.all(q[rows, x.argmax(axis=1)] == 2 ** bits - 1)
    assert s.dtype == np.float32 and z.dtype == np.float32


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_reconstruction_error_bound(bits):
    # |x - x_hat| <= s/2 inside the clamp range (the group's own [min, max]),
    # plus the fp32 rounding of x/s + z (a few ulps of 2^b)
    x = _groups(10 + bits, (500, 64), 3.0)
    q, s, z = O.affine_quantize(x, bits)
    xh = O.affine_dequantize_f64(q, s[:, None], z[:, None])
    slack = s.astype(np.float64)[:, None] * (2.0 ** (bits - 20))
    assert np.all(np.abs(x - xh) <= s.astype(np.float64)[:, None] / 2 + slack)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_rounding_brute_force(bits):
    # every code is the nearest integer of fl(fl(x/s) + z) in [0, 2^b-1], ties to even,
    # found by trying every candidate code
    x = _groups(20 + bits, (40, 9), 2.0)
    q, s, z = O.affine_quantize(x, bits)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            t = float(F32(F32(x[i, j] / s[i]) + z[i]))
            # smallest distance first, then the even code among equally near ones
            best = min((abs(t - c), c % 2, c) for c in range(2 ** bits))
            assert q[i, j] == best[2], (i, j, t, q[i, j], best)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_on_grid_values_reconstruct_exactly(bits):
    # power-of-two s and an integer zero-point: a group holding codes 0 and 2^b-1
    # (so that min/max fix s and z) reconstructs exactly
    levels = 2 ** bits - 1
    rng = np.random.default_rng(bits)
    for s0 in (2.0 ** -3, 0.5, 4.0):
        z0 = int(rng.integers(0, levels + 1))
        codes = rng.integers(0, levels + 1, size=30)
        codes[0], codes[1] = 0, levels
        x = (s0 * (codes - z0)).astype(F32)
        q, s, z = O.affine_quantize(x, bits)
        assert s == F32(s0) and z == F32(z0)
        assert np.array_equal(q, codes.astype(np.uint8))
        assert np.array_equal(O.affine_dequantize_f32(q, s, z), x)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_ties_round_to_even(bits):
    levels = 2 ** bits - 1
    s0, z0 = 0.25, 1
    ks = np.arange(0, levels)                    # x/s + z = k + 1/2 exactly
    x = np.concatenate([[s0 * (0 - z0), s0 * (levels - z0)], s0 * (ks + 0.5 - z0)]).astype(F32)
    q, s, z = O.affine_quantize(x, bits)
    assert s == F32(s0) and z == F32(z0)
    expect = np.where(ks % 2 == 0, ks, ks + 1)
    assert np.array_equal(q[2:], expect.astype(np.uint8))


def test_constant_group():
    for c in (0.0, -1.5, 3.0e-3):
        x = np.full(16, c, F32)
        q, s, z = O.affine_quantize(x, 4)
        assert s == F32(1.0) and np.all(q == 0)
        assert np.array_equal(O.affine_dequantize_f32(q, s, z), x)


def test_key_per_channel_value_per_token_axes():
    # Keys: every channel of every G-token group has its own (s, z);
    # Values: every Gv-slice of every token has its own (s, z).
    spec = O.Spec("int4", d=16, G=8, Gv=4)
    rng = np.random.default_rng(5)
    k = rng.standard_normal((24, 16)).astype(F32)
    k[:, 3] *= 50
    kc, ks, kz, _, _ = O.quantize_key_groups(k, spec)
    assert ks.shape == (3, 16)
    for gi in range(3):
        blk = k[gi * 8:(gi + 1) * 8]
        for c in range(16):
            col = kc[gi * 8:(gi + 1) * 8, c]
            assert col[blk[:, c].argmin()] == 0 and col[blk[:, c].argmax()] == 15
            assert ks[gi, c] == F32(F32(blk[:, c].max() - blk[:, c].min()) / F32(15))
    v = rng.standard_normal((24, 16)).astype(F32)
    vc, vs, vz, _, _ = O.quantize_value_tokens(v, spec)
    assert vs.shape == (24, 4)
    for t in range(24):
        for j in range(4):
            seg = v[t, 4 * j:4 * j + 4]
            cs = vc[t, 4 * j:4 * j + 4]
            assert cs[seg.argmin()] == 0 and cs[seg.argmax()] == 15


# --------------------------------------------------------------------------- #
# FP8 E4M3 (OCP E4M3FN)
# --------------------------------------------------------------------------- #


def test_e4m3_known_values():
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3F: 1.875,
             0x40: 2.0, 0x7E: 448.0, 0x7D: 416.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in cases.items():
        assert O.e4m3_decode(np.array([c]))[0] == v
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF]))).all()
    assert math.copysign(1.0, O.e4m3_decode(np.array([0x80]))[0]) == -1.0


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = O.e4m3_decode(codes).astype(F32)
    assert np.array_equal(O.e4m3_encode(vals), codes)


def _bf16_all_finite():
    bits = np.arange(65536, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)]


def test_e4m3_encode_exhaustive_bf16_brute_force():
    # nearest finite value, ties to the even code, saturate to +-448, keep the sign of zero;
    # found by comparing against every one of the 127 non-negative finite codes
    xs = _bf16_all_finite()
    for scale in (1.0, 0.37, 3.0e-3, 61.0):
        with np.errstate(over="ignore"):
            v = (xs / F32(scale)).astype(F32)
        got = O.e4m3_encode(v)
        table = [(c, float(O.e4m3_decode(np.array([c]))[0])) for c in range(0x7F)]
        a = np.abs(v.astype(np.float64))
        best_d = np.full(a.shape, np.inf)
        best_c = np.zeros(a.shape, np.int64)
        for c, val in table:
            d = np.abs(a - val)
            better = (d < best_d) | ((d == best_d) & (c % 2 == 0))
            best_d = np.where(better, d, best_d)
            best_c = np.where(better, c, best_c)
        best_c = np.where(a > 448.0, 0x7E, best_c)
        best_c |= np.signbit(v).astype(np.int64) << 7
        assert np.array_equal(got, best_c.astype(np.uint8)), scale


def test_fp8_tensor_scale():
    x = np.array([-3.5, 1.0, 2.0], F32)
    assert O.fp8_tensor_scale(x) == F32(F32(3.5) / F32(448))
    assert O.fp8_tensor_scale(np.zeros(4, F32)) == F32(1.0)
    # the calibration tensor's amax maps to the largest finite code
    s = O.fp8_tensor_scale(x)
    assert O.fp8_quantize(x, s)[0] == 0xFE


# --------------------------------------------------------------------------- #
# FP8 E5M2 (OCP E5M2: the high byte of an IEEE binary16)
# --------------------------------------------------------------------------- #


def _f16_of_e5m2(codes):
    """Independent decoder: an E5M2 code is the top byte of a binary16 whose low byte is zero."""
    return (np.asarray(codes, np.uint16) << 8).view(np.float16).astype(np.float64)


def test_e5m2_known_values():
    cases = {0x00: 0.0, 0x01: 2.0 ** -16, 0x03: 3 * 2.0 ** -16, 0x04: 2.0 ** -14, 0x3C: 1.0, 0x3D: 1.25,
             0x3F: 1.75, 0x40: 2.0, 0x7B: 57344.0, 0x7A: 49152.0, 0xBC: -1.0, 0xFB: -57344.0}
    for c, v in cases.items():
        assert O.e5m2_decode(np.array([c]))[0] == v
    assert O.e5m2_decode(np.array([0x7C]))[0] == np.inf and O.e5m2_decode(np.array([0xFC]))[0] == -np.inf
    assert np.isnan(O.e5m2_decode(np.array([0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]))).all()
    assert math.copysign(1.0, O.e5m2_decode(np.array([0x80]))[0]) == -1.0


def test_e5m2_decode_matches_binary16_all_codes():
    codes = np.arange(256)
    a, b = O.e5m2_decode(codes), _f16_of_e5m2(codes)
    same = (a == b) | (np.isnan(a) & np.isnan(b))
    assert same.all()
    num = ~np.isnan(a)
    assert np.array_equal(np.signbit(a[num]), np.signbit(b[num]))


def test_e5m2_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) < 0x7C], dtype=np.uint8)
    vals = O.e5m2_decode(codes).astype(F32)
    assert np.array_equal(O.e5m2_encode(vals), codes)


def test_e5m2_encode_exhaustive_bf16_brute_force():
    # nearest finite value, ties to the even code, saturate to +-57344, keep the sign of zero;
    # candidates decoded by the independent binary16 route
    xs = _bf16_all_finite()
    table = [(c, float(_f16_of_e5m2(np.array([c]))[0])) for c in range(0x7C)]
    for scale in (1.0, 0.37, 3.0e-3, 61.0, 1.0e-6):
        with np.errstate(over="ignore"):
            v = (xs / F32(scale)).astype(F32)
        got = O.e5m2_encode(v)
        a = np.abs(v.astype(np.float64))
        best_d = np.full(a.shape, np.inf)
        best_c = np.zeros(a.shape, np.int64)
        for c, val in table:
            d = np.abs(a - val)
            better = (d < best_d) | ((d == best_d) & (c % 2 == 0))
            best_d = np.where(better, d, best_d)
            best_c = np.where(better, c, best_c)
        best_c = np.where(a > 57344.0, 0x7B, best_c)
        best_c |= np.signbit(v).astype(np.int64) << 7
        assert np.array_equal(got, best_c.astype(np.uint8)), scale


def test_e5m2_tensor_scale():
    x = np.array([-3.5, 1.0, 2.0], F32)
    assert O.fp8_tensor_scale(x, "fp8_e5m2") == F32(F32(3.5) / F32(57344))
    assert O.fp8_tensor_scale(np.zeros(4, F32), "fp8_e5m2") == F32(1.0)
    s = O.fp8_tensor_scale(x, "fp8_e5m2")
    assert O.fp8_quantize(x, s, "fp8_e5m2")[0] == 0xFB
    # E5M2 keeps two mantissa bits: 1 + 1/8 lies halfway between 1 and 1.25 and goes to the even code (1.0)
    assert O.fp8_quantize(np.array([1.125], F32), F32(1.0), "fp8_e5m2")[0] == 0x3C
    assert O.fp8_quantize(np.array([1.375], F32), F32(1.0), "fp8_e5m2")[0] == 0x3E


# --------------------------------------------------------------------------- #
# cache state machine
# --------------------------------------------------------------------------- #


def test_token_split_workloads():
    assert O.token_split(512, O.Spec("int4", G=32, Gv=128, R=32, S=0)) == (0, 480, 32)
    assert O.token_split(8192, O.Spec("int4", G=128, Gv=128, R=128, S=0)) == (0, 8064, 128)
    sp = O.Spec("int2", G=32, Gv=32, R=128, S=0)
    assert O.token_split(32767, sp) == (0, 32608, 159)
    assert O.token_split(32768, sp) == (0, 32640, 128)
    sp5 = O.Spec("int4", G=16, Gv=128, R=64, S=1)
    assert O.token_split(1, sp5) == (1, 0, 0)
    assert O.token_split(80, sp5) == (1, 0, 79)
    assert O.token_split(81, sp5) == (1, 16, 64)
    assert O.token_split(9, O.Spec("fp8_e4m3", G=1, R=0, S=0)) == (0, 9, 0)
    assert O.token_split(9, O.Spec("fp8_e5m2", G=1, R=0, S=2)) == (2, 7, 0)
    # a skip layer never quantizes, however long the sequence
    assert O.token_split(100000, O.Spec("bf16", G=16, R=0, S=1)) == (1, 0, 99999)


def _same_cache(a, b):
    for f in ("sink_k", "sink_v", "k_codes", "v_codes", "resid_k", "resid_v", "k_s", "k_z", "v_s", "v_z",
              "k_sp_idx", "k_sp_val", "v_sp_idx", "v_sp_val"):
        x, y = getattr(a, f), getattr(b, f)
        if x is None:
            assert y is None
            continue
        assert x.shape == y.shape and np.array_equal(x, y), f


@pytest.mark.parametrize("spec", [
    O.Spec("int4", d=16, G=8, Gv=8, R=4, S=0),
    O.Spec("int2", d=16, G=4, Gv=16, R=8, S=1),
    O.Spec("int8", d=16, G=16, Gv=4, R=0, S=2),
    O.Spec("fp8_e4m3", d=16, G=1, Gv=16, R=0, S=1),
    O.Spec("fp8_e5m2", d=16, G=1, Gv=16, R=0, S=0),
    O.Spec("bf16", d=16, G=16, Gv=16, R=0, S=1),
    O.Spec("int4", d=16, G=8, Gv=8, R=4, S=1, k_outliers=2, v_outliers=1),
    O.Spec("int2", d=16, G=4, Gv=16, R=8, S=0, k_outliers=1, v_outliers=3),
])
def test_bulk_build_equals_appends(spec):
    rng = np.random.default_rng(7)
    T = 61
    k = rng.standard_normal((T, 16)).astype(F32)
    v = rng.standard_normal((T, 16)).astype(F32)
    ks = O.fp8_tensor_scale(k, spec.fmt) if spec.is_fp8 else None
    vs = O.fp8_tensor_scale(v, spec.fmt) if spec.is_fp8 else None
    hc = O.empty_head_cache(spec, ks, vs)
    for t in range(T):
        O.append_token(hc, k[t], v[t])
        bulk = O.build_head_cache(k[:t + 1], v[:t + 1], spec, ks, vs)
        _same_cache(hc, bulk)
        n_sink, qn, r = O.token_split(t + 1, spec)
        assert (len(hc.sink_k), len(hc.k_codes), len(hc.resid_k)) == (n_sink, qn, r)
        if spec.is_bf16:
            assert qn == 0 and np.array_equal(hc.resid_k, k[min(t + 1, spec.S):t + 1])
        elif not spec.is_fp8:
            assert r < spec.R + spec.G


# --------------------------------------------------------------------------- #
# attention
# --------------------------------------------------------------------------- #


def _brute_attention(q, K, V, scale):
    """Plain-Python softmax(q K^T * scale) V and its log-sum-exp."""
    scores = [sum(float(a) * float(b) for a, b in zip(q, krow)) * scale for krow in K]
    mx = max(scores)
    w = [math.exp(s - mx) for s in scores]
    tot = sum(w)
    out = [sum(w[t] * float(V[t][c]) for t in range(len(V))) / tot for c in range(len(V[0]))]
    return out, mx + math.log(tot)


def _dequant_brute(hc):
    """x_hat = s (q - z) element by element in Python floats (fp64)."""
    sp = hc.spec
    ks, vs = [], []
    for t in range(len(hc.sink_k)):
        ks.append(list(map(float, hc.sink_k[t])))
        vs.append(list(map(float, hc.sink_v[t])))
    for t in range(len(hc.k_codes)):
        if sp.fmt == "fp8_e5m2":
            ks.append([float(hc.k_scale) * float(_f16_of_e5m2(np.array([c]))[0]) for c in hc.k_codes[t]])
            vs.append([float(hc.v_scale) * float(_f16_of_e5m2(np.array([c]))[0]) for c in hc.v_codes[t]])
        elif sp.is_fp8:
            ks.append([float(hc.k_scale) * float(O.e4m3_decode(np.array([c]))[0]) for c in hc.k_codes[t]])
            vs.append([float(hc.v_scale) * float(O.e4m3_decode(np.array([c]))[0]) for c in hc.v_codes[t]])
        else:
            g = t // sp.G
            ks.append([float(hc.k_s[g, c]) * (int(hc.k_codes[t, c]) - float(hc.k_z[g, c])) for c in range(sp.d)])
            vs.append([float(hc.v_s[t, c // sp.Gv]) * (int(hc.v_codes[t, c]) - float(hc.v_z[t, c // sp.Gv]))
                       for c in range(sp.d)])
            for j in range(sp.k_outliers):  # the kept outliers add at their channels
                ks[-1][int(hc.k_sp_idx[t, j])] += float(hc.k_sp_val[t, j])
            for j in range(sp.v_outliers):
                vs[-1][int(hc.v_sp_idx[t, j])] += float(hc.v_sp_val[t, j])
    for t in range(len(hc.resid_k)):
        ks.append(list(map(float, hc.resid_k[t])))
        vs.append(list(map(float, hc.resid_v[t])))
    return ks, vs


@pytest.mark.parametrize("spec", [
    O.Spec("int4", d=16, G=8, Gv=8, R=4, S=1),
    O.Spec("int2", d=16, G=4, Gv=16, R=8, S=0),
    O.Spec("int8", d=16, G=16, Gv=4, R=2, S=0),
    O.Spec("fp8_e4m3", d=16, G=1, Gv=16, R=0, S=1),
    O.Spec("fp8_e5m2", d=16, G=1, Gv=16, R=0, S=0),
    O.Spec("bf16", d=16, G=16, Gv=16, R=0, S=1),
    O.Spec("int4", d=16, G=8, Gv=8, R=4, S=1, k_outliers=2, v_outliers=2),
    O.Spec("int8", d=16, G=16, Gv=4, R=0, S=0, k_outliers=1, v_outliers=4),
])
def test_attention_brute_force(spec):
    rng = np.random.default_rng(11)
    B, Hkv, g, T = 2, 2, 3, 37
    q = rng.standard_normal((B, Hkv * g, 16)).astype(F32)
    caches = []
    for b in range(B):
        row = []
        for h in range(Hkv):
            k = (rng.standard_normal((T, 16)) * 2).astype(F32)
            v = rng.standard_normal((T, 16)).astype(F32)
            ks = O.fp8_tensor_scale(k, spec.fmt) if spec.is_fp8 else None
            vs = O.fp8_tensor_scale(v, spec.fmt) if spec.is_fp8 else None
            row.append(O.build_head_cache(k, v, spec, ks, vs))
        caches.append(row)
    out, lse = O.decode_attention(q, caches)
    for b in range(B):
        for hq in range(Hkv * g):
            K, V = _dequant_brute(caches[b][hq // g])
            o, l = _brute_attention(q[b, hq], K, V, 1 / math.sqrt(16))
            assert np.allclose(out[b, hq], o, rtol=0, atol=1e-12)
            assert abs(lse[b, hq] - l) < 1e-12


@pytest.mark.parametrize("spec", [
    O.Spec("int4", d=16, G=8, Gv=8, R=4, S=1),
    O.Spec("fp8_e4m3", d=16, G=1, Gv=16, R=0, S=0),
    O.Spec("bf16", d=16, G=16, Gv=16, R=0, S=1),
])
def test_multi_query_causal_brute_force(spec):
    # query i of M sees tokens 0 .. T - M + i of the full cache; checked against the
    # plain-Python attention over that prefix of the element-wise dequantized tokens
    rng = np.random.default_rng(5)
    B, Hkv, g, M = 2, 2, 2, 3
    lens = [23, 2]  # the second sequence is shorter than M: its first query sees nothing
    caches = []
    for b in range(B):
        row = []
        for h in range(Hkv):
            k = rng.standard_normal((lens[b], 16)).astype(F32)
            v = rng.standard_normal((lens[b], 16)).astype(F32)
            ks = O.fp8_tensor_scale(k, spec.fmt) if spec.is_fp8 else None
            vs = O.fp8_tensor_scale(v, spec.fmt) if spec.is_fp8 else None
            row.append(O.build_head_cache(k, v, spec, ks, vs))
        caches.append(row)
    q = rng.standard_normal((B, M, Hkv * g, 16)).astype(F32)
    out, lse = O.decode_attention_multi(q, caches)
    for b in range(B):
        for i in range(M):
            n = lens[b] - M + i + 1
            for hq in range(Hkv * g):
                K, V = _dequant_brute(caches[b][hq // g])
                if n <= 0:
                    assert np.all(out[b, i, hq] == 0) and lse[b, i, hq] == -math.inf
                    continue
                o, l = _brute_attention(q[b, i, hq], K[:n], V[:n], 1 / math.sqrt(16))
                assert np.allclose(out[b, i, hq], o, rtol=0, atol=1e-12)
                assert abs(lse[b, i, hq] - l) < 1e-12
    # one query token is the plain decode step
    o1, l1 = O.decode_attention_multi(q[:, -1:], caches)
    o2, l2 = O.decode_attention(q[:, -1], caches)
    assert np.array_equal(o1[:, 0], o2) and np.array_equal(l1[:, 0], l2)


def test_attention_single_token_and_uniform():
    spec = O.Spec("int4", d=8, G=4, Gv=8, R=4, S=0)
    k = np.array([[1, -2, 0.5, 0, 3, 1, 1, -1]], F32)
    v = np.array([[0.25, 1, -1, 2, 0, 0, 3, 4]], F32)
    hc = O.build_head_cache(k, v, spec)
    q = np.ones((1, 1, 8), F32)
    out, lse = O.decode_attention(q, [[hc]])
    assert np.allclose(out[0, 0], v[0], atol=0, rtol=0)
    assert lse[0, 0] == pytest.approx(float(k[0] @ q[0, 0]) / math.sqrt(8), abs=1e-15)
    # every token has the same key -> every score equal: out = mean(v), lse = score + ln T
    T = 6
    kk = np.repeat(k, T, axis=0)
    vv = np.arange(T * 8, dtype=F32).reshape(T, 8)
    hc = O.build_head_cache(kk, vv, spec)
    assert len(hc.k_codes) == 0                     # T < R + G: all bf16
    out, lse = O.decode_attention(q, [[hc]])
    assert np.allclose(out[0, 0], vv.mean(axis=0), atol=1e-12)
    assert lse[0, 0] == pytest.approx(float(k[0] @ q[0, 0]) / math.sqrt(8) + math.log(T), abs=1e-12)


def test_gqa_equals_replicated_mha_and_token_order():
    spec = O.Spec("int4", d=16, G=8, Gv=16, R=8, S=0)
    rng = np.random.default_rng(3)
    T = 40
    k = rng.standard_normal((T, 16)).astype(F32)
    v = rng.standard_normal((T, 16)).astype(F32)
    hc = O.build_head_cache(k, v, spec)
    q = rng.standard_normal((1, 4, 16)).astype(F32)
    out_gqa, lse_gqa = O.decode_attention(q, [[hc]])
    out_mha, lse_mha = O.decode_attention(q, [[hc, hc, hc, hc]])
    assert np.array_equal(out_gqa, out_mha) and np.array_equal(lse_gqa, lse_mha)
    kh, vh = O.dequantized_f64(hc)
    perm = rng.permutation(T)
    for j in range(4):
        o1, l1 = O.attend_head(q[0, j], kh, vh, 0.25)
        o2, l2 = O.attend_head(q[0, j], kh[perm], vh[perm], 0.25)
        assert np.allclose(o1, o2, atol=1e-13) and abs(l1 - l2) < 1e-13


# --------------------------------------------------------------------------- #
# the fp32 cache export (dequantized_f32): what kvq_dequantize is compared with
# "KV Cache Quantization Analysis", section 2 (x_hat = s(q - z)); section 4 (FP8 value times its scale)
# --------------------------------------------------------------------------- #


def _on_grid_groups(bits, qn, d, G, Gv, seed):
    """K and V of qn quantized tokens where every quantization group lies on a grid of its own:
    s a power of two and z an integer, different for every group, and the group holds the
    codes 0 and 2^b - 1 (at positions that move with the group).  Every value is s (q - z) with
    |q - z| < 256, so it is exact in bf16 and fp32.  Returns (k, v, k_s, k_z, v_s, v_z)."""
    rng = np.random.default_rng(seed)
    L = 2 ** bits - 1
    nk = qn // G
    k_s = np.empty((nk, d)); k_z = np.empty((nk, d))
    v_s = np.empty((qn, d // Gv)); v_z = np.empty((qn, d // Gv))
    kq = rng.integers(0, L + 1, size=(qn, d))
    vq = rng.integers(0, L + 1, size=(qn, d))
    for j in range(nk):
        for c in range(d):
            k_s[j, c] = 2.0 ** -(1 + (c + 2 * j) % 4)
            k_z[j, c] = (5 * c + 3 * j + 1) % (L + 1)
            lo, hi = j * G + (c % G), j * G + ((c + 1) % G)
            kq[lo, c], kq[hi, c] = 0, L
    for t in range(qn):
        for j in range(d // Gv):
            v_s[t, j] = 2.0 ** -(1 + (t + 3 * j) % 4)
            v_z[t, j] = (3 * t + 7 * j + 2) % (L + 1)
            lo, hi = j * Gv + (t % Gv), j * Gv + ((t + 1) % Gv)
            vq[t, lo], vq[t, hi] = 0, L
    gk = np.arange(qn) // G
    k = (k_s[gk] * (kq - k_z[gk])).astype(F32)
    v = (np.repeat(v_s, Gv, axis=1) * (vq - np.repeat(v_z, Gv, axis=1))).astype(F32)
    return k, v, k_s, k_z, v_s, v_z


@pytest.mark.parametrize("bits,G,Gv,R,S", [(2, 8, 16, 5, 1), (4, 16, 32, 3, 2), (8, 4, 8, 7, 0)])
def test_dequantized_f32_returns_on_grid_inputs_in_token_order(bits, G, Gv, R, S):
    d, n_groups = 32, 3
    qn = n_groups * G
    kq, vq, k_s, k_z, v_s, v_z = _on_grid_groups(bits, qn, d, G, Gv, seed=bits)
    rng = np.random.default_rng(100 + bits)
    # sink and residual tokens: arbitrary bf16 values, distinct from the grid values
    sink_k, sink_v = (O.bf16_to_f32(rng.integers(0x3F80, 0x4100, size=(S, d)).astype(np.uint16)) for _ in range(2))
    res_k, res_v = (O.bf16_to_f32(rng.integers(0xC000, 0xC100, size=(R, d)).astype(np.uint16)) for _ in range(2))
    k = np.concatenate([sink_k, kq, res_k]).astype(F32)
    v = np.concatenate([sink_v, vq, res_v]).astype(F32)
    spec = O.Spec(f"int{bits}", d=d, G=G, Gv=Gv, R=R, S=S)
    assert O.token_split(len(k), spec) == (S, qn, R)
    hc = O.build_head_cache(k, v, spec)
    # the quantizer recovers every group's grid exactly ...
    assert np.array_equal(hc.k_s, k_s.astype(F32)) and np.array_equal(hc.k_z, k_z.astype(F32))
    assert np.array_equal(hc.v_s, v_s.astype(F32)) and np.array_equal(hc.v_z, v_z.astype(F32))
    # ... and the export returns the inputs themselves, bit for bit, sink first, residual last
    ko, vo = O.dequantized_f32(hc)
    assert ko.dtype == np.float32 and vo.dtype == np.float32
    assert np.array_equal(ko.view(np.uint32), k.view(np.uint32))
    assert np.array_equal(vo.view(np.uint32), v.view(np.uint32))


@pytest.mark.parametrize("fmt,codes,k_scale,v_scale,k_expect,v_expect", [
    # E4M3: 0x38 = 1.0, 0x7E = 448 (largest finite), 0x01 = 2^-9 (smallest subnormal), 0xB8 = -1.0, +-0
    ("fp8_e4m3", [0x38, 0x7E, 0x01, 0xB8, 0x00, 0x80], 0.5, 2.0,
     [0.5, 224.0, 2.0 ** -10, -0.5, 0.0, -0.0], [2.0, 896.0, 2.0 ** -8, -2.0, 0.0, -0.0]),
    # E5M2: 0x3C = 1.0, 0x7B = 57344 (largest finite), 0x01 = 2^-16, 0xBC = -1.0, 0x46 = 6.0
    ("fp8_e5m2", [0x3C, 0x7B, 0x01, 0xBC, 0x46], 0.25, 4.0,
     [0.25, 14336.0, 2.0 ** -18, -0.25, 1.5], [4.0, 229376.0, 2.0 ** -14, -4.0, 24.0]),
])
def test_dequantized_f32_fp8_worked_values(fmt, codes, k_scale, v_scale, k_expect, v_expect):
    d = 4
    spec = O.Spec(fmt, d=d, G=1, Gv=d, R=0, S=1)
    n = len(codes)
    cm = np.array([[c] * d for c in codes], np.uint8)           # token t: code codes[t] in every channel
    sink = np.full((1, d), 3.0, F32)
    hc = O.HeadCache(spec, sink.copy(), -sink, cm, cm[::-1].copy(), np.zeros((0, d), F32), np.zeros((0, d), F32),
                     k_scale=F32(k_scale), v_scale=F32(v_scale))
    ko, vo = O.dequantized_f32(hc)
    assert ko.shape == (1 + n, d) and ko.dtype == np.float32
    assert np.array_equal(ko[0], sink[0]) and np.array_equal(vo[0], -sink[0])
    want_k = np.array(k_expect, F32)
    want_v = np.array(v_expect, F32)[::-1]
    assert np.array_equal(ko[1:, 0].view(np.uint32), want_k.view(np.uint32))   # sign of zero included
    assert np.array_equal(vo[1:, 0].view(np.uint32), want_v.view(np.uint32))
    assert np.all(ko[1:] == ko[1:, :1]) and np.all(vo[1:] == vo[1:, :1])


# --------------------------------------------------------------------------- #
# pre-RoPE Keys ("KV Cache Quantization Analysis", section 3 RoPE bullet; section 4 KVQuant (ii))
# --------------------------------------------------------------------------- #


def _rope_brute(x, t, base):
    """Rotate-half RoPE of one vector at position t, plain Python (math.cos / math.sin)."""
    d = len(x)
    h = d // 2
    out = [0.0] * d
    for i in range(h):
        a = t * base ** (-(2 * i) / d)
        out[i] = float(x[i]) * math.cos(a) - float(x[i + h]) * math.sin(a)
        out[i + h] = float(x[i + h]) * math.cos(a) + float(x[i]) * math.sin(a)
    return out


def test_rope_closed_forms():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((6, 16))
    base = 10000.0
    # position 0 is the identity
    assert np.array_equal(O.rope_rotate(x, np.zeros(6), base), x)
    # a rotation by t then by -t is the identity; every channel pair keeps its norm
    t = np.array([1, 5, 17, 300, 4095, 65535], dtype=np.float64)
    y = O.rope_rotate(x, t, base)
    assert np.allclose(O.rope_rotate(y, -t, base), x, rtol=0, atol=1e-12)
    assert np.allclose(y[:, :8] ** 2 + y[:, 8:] ** 2, x[:, :8] ** 2 + x[:, 8:] ** 2, rtol=0, atol=1e-12)
    # the score of a rotated query and a rotated key depends only on their distance
    q, k = rng.standard_normal((1, 16)), rng.standard_normal((1, 16))
    def score(m, n):
        return float((O.rope_rotate(q, [m], base) @ O.rope_rotate(k, [n], base).T)[0, 0])
    for m, n in ((5, 2), (40, 37), (1003, 1000)):
        assert abs(score(m, n) - score(3, 0)) < 1e-12
    assert abs(score(7, 7) - float((q @ k.T)[0, 0])) < 1e-12
    # the pairing and the angles against a plain-Python rotation (d = 8)
    x8 = rng.standard_normal(8)
    for tt in (0, 1, 9, 1234):
        assert np.allclose(O.rope_rotate(x8[None], [tt], 500000.0)[0], _rope_brute(x8, tt, 500000.0), rtol=0,
                           atol=1e-12)


@pytest.mark.parametrize("spec", [
    O.Spec("int4", d=16, G=8, Gv=8, R=4, S=1, rope_base=10000.0),
    O.Spec("int8", d=16, G=16, Gv=4, R=2, S=0, rope_base=500000.0),
    O.Spec("int2", d=16, G=4, Gv=16, R=8, S=2, rope_base=10000.0),
])
def test_attention_over_pre_rope_keys_brute_force(spec):
    # every dequantized Key (sink, quantized, residual) is rotated at its own position
    rng = np.random.default_rng(13)
    B, Hkv, g, T = 2, 2, 3, 37
    q = rng.standard_normal((B, Hkv * g, 16)).astype(F32)
    caches = [[O.build_head_cache((rng.standard_normal((T, 16)) * 2).astype(F32),
                                  rng.standard_normal((T, 16)).astype(F32), spec) for _ in range(Hkv)]
              for _ in range(B)]
    out, lse = O.decode_attention(q, caches)
    for b in range(B):
        for hq in range(Hkv * g):
            K, V = _dequant_brute(caches[b][hq // g])
            K = [_rope_brute(K[t], t, spec.rope_base) for t in range(T)]
            o, l = _brute_attention(q[b, hq], K, V, 1 / math.sqrt(16))
            assert np.allclose(out[b, hq], o, rtol=0, atol=1e-11)
            assert abs(lse[b, hq] - l) < 1e-11
    # the stored cache is the same as without RoPE (Keys quantized before the rotation)
    plain = O.Spec(spec.fmt, d=16, G=spec.G, Gv=spec.Gv, R=spec.R, S=spec.S)
    k = rng.standard_normal((T, 16)).astype(F32)
    v = rng.standard_normal((T, 16)).astype(F32)
    _same_cache(O.build_head_cache(k, v, spec), O.build_head_cache(k, v, plain))



# --------------------------------------------------------------------------- #
# dense-and-sparse outliers ("KV Cache Quantization Analysis", section 4, KVQuant (iv); section 2 outliers)
# --------------------------------------------------------------------------- #


def _top_n_brute(row, n):
    """Channels of the n largest |x| of a row, ties to the lower channel, plain Python; ascending."""
    chosen = []
    for _ in range(n):
        best = None
        for c in range(len(row)):
            if c in chosen:
                continue
            if best is None or abs(float(row[c])) > abs(float(row[best])):
                best = c
        chosen.append(best)
    return sorted(chosen)


def test_outlier_selection_brute_force():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((40, 16)).astype(F32)
    x[3, [2, 9, 14]] = 5.0            # ties at the top: the lower channels win
    x[4, :] = 0.0                     # an all-zero row: channels 0 .. n-1
    x[5, [1, 7]] = [-3.0, 3.0]        # equal magnitudes, opposite signs
    for n in (0, 1, 2, 3, 5):
        dense, idx, val = O.split_outliers(x, n)
        for i in range(len(x)):
            want = _top_n_brute(x[i], n)
            assert list(idx[i]) == want, (n, i)
            assert np.array_equal(val[i], x[i, want])
            d = x[i].copy()
            d[want] = 0.0
            assert np.array_equal(dense[i], d)


@pytest.mark.parametrize("bits,nk,nv", [(2, 1, 2), (4, 2, 1), (8, 3, 3)])
def test_outliers_reconstruct_exactly_on_grid(bits, nk, nv):
    # dense rows on a grid of their own per group (power-of-two s, integer z, codes 0 and 2^b - 1
    # present), planted outliers far above every dense value at positions that are neither a group's
    # minimum nor its maximum and hold the code z (dense value 0): the split recovers the planted
    # outliers and the export returns the inputs exactly
    d, G, Gv, n_groups = 32, 8, 16, 2
    qn = n_groups * G
    L = 2 ** bits - 1
    rng = np.random.default_rng(40 + bits)
    kq = rng.integers(0, L + 1, size=(qn, d))
    vq = rng.integers(0, L + 1, size=(qn, d))
    k_s, k_z = np.empty((n_groups, d)), rng.integers(1, L, size=(n_groups, d))
    v_s, v_z = np.empty((qn, d // Gv)), rng.integers(1, L, size=(qn, d // Gv))
    reserved_k = np.zeros((qn, d), bool)   # group minimum / maximum positions
    reserved_v = np.zeros((qn, d), bool)
    for j in range(n_groups):
        for c in range(d):
            k_s[j, c] = 2.0 ** -(1 + (c + j) % 3)
            lo, hi = j * G + (c % G), j * G + ((c + 1) % G)
            kq[lo, c], kq[hi, c] = 0, L
            reserved_k[lo, c] = reserved_k[hi, c] = True
    for t in range(qn):
        for j in range(d // Gv):
            v_s[t, j] = 2.0 ** -(1 + (t + j) % 3)
            lo, hi = j * Gv + (t % Gv), j * Gv + ((t + 1) % Gv)
            vq[t, lo], vq[t, hi] = 0, L
            reserved_v[t, lo] = reserved_v[t, hi] = True
    gk = np.arange(qn) // G
    kidx = np.sort(np.stack([rng.choice(np.flatnonzero(~reserved_k[t]), nk, replace=False) for t in range(qn)]), 1)
    vidx = np.sort(np.stack([rng.choice(np.flatnonzero(~reserved_v[t]), nv, replace=False) for t in range(qn)]), 1)
    rows = np.arange(qn)[:, None]
    kq[rows, kidx] = k_z[gk[:, None], kidx]                     # dense value 0 there
    vq[rows, vidx] = np.repeat(v_z, Gv, axis=1)[rows, vidx]
    kd = (k_s[gk] * (kq - k_z[gk])).astype(F32)
    vd = (np.repeat(v_s, Gv, axis=1) * (vq - np.repeat(v_z, Gv, axis=1))).astype(F32)
    assert np.all(kd[rows, kidx] == 0) and np.all(vd[rows, vidx] == 0) and np.abs(kd).max() < 200
    kval = (rng.integers(200, 400, size=(qn, nk)) * np.where(rng.random((qn, nk)) < 0.5, -1, 1)).astype(F32)
    vval = (rng.integers(200, 400, size=(qn, nv)) * np.where(rng.random((qn, nv)) < 0.5, -1, 1)).astype(F32)
    k, v = kd.copy(), vd.copy()
    k[rows, kidx], v[rows, vidx] = kval, vval
    spec = O.Spec(f"int{bits}", d=d, G=G, Gv=Gv, R=0, S=0, k_outliers=nk, v_outliers=nv)
    hc = O.build_head_cache(k, v, spec)
    assert np.array_equal(hc.k_sp_idx, kidx) and np.array_equal(hc.k_sp_val, kval)
    assert np.array_equal(hc.v_sp_idx, vidx) and np.array_equal(hc.v_sp_val, vval)
    assert np.array_equal(hc.k_s, k_s.astype(F32)) and np.array_equal(hc.k_z, k_z.astype(F32))
    assert np.array_equal(hc.v_s, v_s.astype(F32)) and np.array_equal(hc.v_z, v_z.astype(F32))
    ko, vo = O.dequantized_f32(hc)
    assert np.array_equal(ko.view(np.uint32), k.view(np.uint32)) and np.array_equal(vo.view(np.uint32), v.view(np.uint32))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_outlier_split_error_bound(bits):
    # every entry, kept outlier or not, is within s/2 (of its dense group) of its input
    rng = np.random.default_rng(60 + bits)
    d, G, Gv, qn = 16, 8, 8, 32
    x = (rng.standard_normal((qn, d)) * np.where(rng.random((qn, d)) < 0.05, 30, 1)).astype(F32)
    v = (rng.standard_normal((qn, d)) * np.where(rng.random((qn, d)) < 0.05, 30, 1)).astype(F32)
    spec = O.Spec(f"int{bits}", d=d, G=G, Gv=Gv, k_outliers=2, v_outliers=2)
    hc = O.build_head_cache(x, v, spec)
    kh, vh = O.dequantized_f64(hc)
    ks = np.repeat(hc.k_s, G, axis=0).astype(np.float64)
    vs = np.repeat(hc.v_s, Gv, axis=1).astype(np.float64)
    assert np.all(np.abs(kh - x) <= ks / 2 * (1 + 1e-5) + 1e-30)
    assert np.all(np.abs(vh - v) <= vs / 2 * (1 + 1e-5) + 1e-30)
    # the split narrows the grids: the dense scales never exceed those of the plain quantizer
    plain = O.build_head_cache(x, v, O.Spec(f"int{bits}", d=d, G=G, Gv=Gv))
    assert np.all(hc.k_s <= plain.k_s) and np.all(hc.v_s <= plain.v_s)

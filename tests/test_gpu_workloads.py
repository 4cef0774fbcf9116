"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

Each layer is built and stepped exactly as the benchmark does (bench.Layer:
cache of T-1 tokens, one decode step = append of the new token + split pass +
combine; FP8 layers without sink tokens take the step as one
kvq_append_decode_attention launch).  The oracle then rebuilds sampled (sequence, kv head) pairs from the
same seeded inputs and checks, for those pairs:
  * the dequantized export (codes, scales, zero-points, bf16 parts): bit-exact;
  * attention outputs of all query heads of the pair: fp32 within
    2e-3 * max|ref| (over the sampled heads), lse within 1e-4; the bf16 output
    the benchmark writes equals the RNE of the fp32 output.
Inputs come from the seeded device generator; the oracle receives copies of
those inputs, never anything the CUDA path computed.
"""
import math

import numpy as np
import pytest

from oracle import kvq_oracle as O
from quantized_kv_cache_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bench  # noqa: E402
import kvq_testlib as TL  # noqa: E402
from quantized_kv_cache_decode_gb300 import kvq  # noqa: E402

DEV = torch.device("cuda", 0)


def _spec(fmt):
    fp8 = bench.is_fp8(fmt)
    return O.Spec(fmt.fmt, d=128, G=1 if fp8 else fmt.G, Gv=fmt.Gv, R=0 if fp8 else fmt.R, S=fmt.S,
                  rope_base=fmt.rope_base, k_outliers=fmt.k_outliers, v_outliers=fmt.v_outliers)


def _pairs(w, n, seed):
    # n seeded (sequence, kv head) pairs, always with the first and the last pair, and for ragged
    # batches the shortest and the longest sequence
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (w.batch - 1, w.num_kv_heads - 1)}
    if w.seq_len_range is not None:
        lens = I.seq_lens(w)
        pairs |= {(int(np.argmin(lens)), 1 % w.num_kv_heads), (int(np.argmax(lens)), 2 % w.num_kv_heads)}
    while len(pairs) < n:
        pairs.add((int(rng.integers(w.batch)), int(rng.integers(w.num_kv_heads))))
    return sorted(pairs)


def _check_layer(w, l, pairs, seed_offset=0):
    fmt = w.layer_formats[l]
    spec = _spec(fmt)
    n_app = max(1, w.append_tokens)
    lens_after = I.seq_lens(w) + w.append_tokens if w.seq_len_range is not None else np.full(w.batch, w.seq_len)
    lens_before = [int(t) - n_app for t in lens_after]
    lay = bench.Layer(kvq, torch, w, l, fmt, lens_before, n_app, DEV, seed_offset=seed_offset)
    # one benchmark step (the calls the bench makes: FP8 layers without sink tokens in one
    # kvq_append_decode_attention launch, the others append then decode)
    lay.step_calls()
    torch.cuda.synchronize()
    assert lay.status.item() == 0
    out16 = lay.out.clone()
    # the same cache, fp32 output
    M = w.n_query
    rows = (lay.B, lay.Hq) if M == 1 else (lay.B, M, lay.Hq)
    out32 = torch.empty(rows + (128,), dtype=torch.float32, device=DEV)
    lse32 = torch.empty(rows, dtype=torch.float32, device=DEV)
    if M == 1:
        kvq.decode_attention(lay.cfg, lay.struct, lay.q, lay.Hq, lay.lens_after, lay.B, lay.scale, out32, False,
                             lse32, lay.ws, lay.wsb, lay.status)
    else:
        kvq.decode_attention_multi(lay.cfg, lay.struct, lay.q, M, lay.Hq, lay.lens_after, lay.B, lay.scale, out32,
                                   False, lse32, lay.ws, lay.wsb, lay.status)
    torch.cuda.synchronize()
    assert torch.equal(out16, out32.to(torch.bfloat16))
    assert torch.equal(lay.lse, lse32)
    q = lay.q.float().cpu().numpy()
    # the oracle's inputs: the seeded draws, regenerated and copied to the host
    uniform = w.seq_len_range is None
    ks = vs = None
    if uniform:
        kd, vd = I.device_kv_bf16(w, l, int(lens_after[0]), DEV, batch=w.batch, seed_offset=seed_offset)
        if spec.is_fp8:
            kall = kd.float().cpu().numpy()
            vall = vd.float().cpu().numpy()
            ks, vs = O.fp8_tensor_scale(kall, spec.fmt), O.fp8_tensor_scale(vall, spec.fmt)
            del kall, vall
            assert lay.cache.k_tensor_scale.item() == float(ks)
            assert lay.cache.v_tensor_scale.item() == float(vs)
    refs, outs, lses, olses = [], [], [], []
    for b, h in pairs:
        T = int(lens_after[b])
        if uniform:
            k = kd[b, h].float().cpu().numpy()
            v = vd[b, h].float().cpu().numpy()
        else:
            wb = I.Workload(**{**w.__dict__, "batch": 1})
            k1, v1 = I.device_kv_bf16(wb, l, T, DEV, batch=1, seed_offset=seed_offset + 7 * b)
            k, v = k1[0, h].float().cpu().numpy(), v1[0, h].float().cpu().numpy()
        hc = O.build_head_cache(k[:T - n_app], v[:T - n_app], spec, ks, vs)
        for t in range(T - n_app, T):
            O.append_token(hc, k[t], v[t])
        # dequantized export of this sequence, bit-exact
        ko = torch.empty((1, w.num_kv_heads, T, 128), dtype=torch.float32, device=DEV)
        vo = torch.empty_like(ko)
        kvq.dequantize(lay.cfg, lay.cache.seq_struct(b), lay.lens_after[b:b + 1], 1, T, ko, vo, lay.status)
        torch.cuda.synchronize()
        kr, vr = O.dequantized_f32(hc)
        assert np.array_equal(ko[0, h].cpu().numpy().view(np.uint32), kr.view(np.uint32)), (b, h)
        assert np.array_equal(vo[0, h].cpu().numpy().view(np.uint32), vr.view(np.uint32)), (b, h)
        kh, vh = O.attention_keys(hc)  # (pre-RoPE layers: Keys rotated at their positions)
        for m in range(M):
            n = T - M + m + 1  # query token m attends to its causal prefix
            for j in range(w.gqa):
                hq = h * w.gqa + j
                qv, ov, lv = (q[b, hq], out32[b, hq], lse32[b, hq]) if M == 1 else \
                    (q[b, m, hq], out32[b, m, hq], lse32[b, m, hq])
                o, ls = O.attend_head(qv, kh[:n], vh[:n], lay.scale)
                refs.append(o)
                olses.append(ls)
                outs.append(ov.cpu().numpy())
                lses.append(lv.item())
    assert lay.status.item() == 0
    TL.check_attention(np.array(outs), np.array(lses), np.array(refs), np.array(olses))


def test_tiny_kivi_int4_all_pairs():
    w = I.tiny_int4()
    _check_layer(w, 0, [(0, 0), (0, 1)])


def test_llama3_8b_fp8_sampled():
    w = I.llama3_8b_fp8()
    _check_layer(w, 0, _pairs(w, 8, 1))


def test_llama3_8b_fp8_e5m2_sampled():
    w = I.llama3_8b_fp8_e5m2()
    _check_layer(w, 0, _pairs(w, 6, 2))


def test_llama3_8b_fp8_two_query_tokens_sampled():
    w = I.llama3_8b_fp8_2q()
    _check_layer(w, 0, _pairs(w, 6, 3))


def test_llama3_8b_bf16_skip_layer_sampled():
    w = I.llama3_8b_bf16_skip()
    _check_layer(w, 0, _pairs(w, 6, 4))


def test_llama3_8b_int4_pre_rope_sampled():
    w = I.llama3_8b_int4_prerope()
    _check_layer(w, 0, _pairs(w, 6, 5))


def test_llama3_8b_int4_dense_and_sparse_sampled():
    w = I.llama3_8b_int4_sparse()
    _check_layer(w, 0, _pairs(w, 6, 6))


@pytest.mark.parametrize("layer", [0, 79])
def test_llama3_70b_int4_sampled(layer):
    w = I.llama3_70b_int4()
    _check_layer(w, layer, _pairs(w, 16, 7 + layer))


def test_llama2_7b_int2_append_spill_sampled():
    w = I.llama2_7b_int2()
    _check_layer(w, 0, _pairs(w, 16, 9))


@pytest.mark.parametrize("layer", [0, 31, 63])
def test_paged_mixed_sampled(layer):
    w = I.paged_mixed()
    _check_layer(w, layer, _pairs(w, 16, 10 + layer))


def test_max_batch_many_short_sequences():
    # the largest batch the library accepts, lengths 0..40 (empty, bf16-only and quantized)
    B = 2048
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 41, size=B)
    lens[:3] = [0, 1, 40]
    gl = TL.GpuLayer("int4", 1, lens, 16, 128, 16, 0, seed=4)
    kb = np.zeros((B, 1, 40, 128), np.uint16)
    vb = np.zeros_like(kb)
    for b in range(B):
        kb[b, 0] = I.random_bf16(b, (40, 128))
        vb[b, 0] = I.random_bf16(b + 10 ** 6, (40, 128))
    # per sequence appends (batch = 1 views)
    for b in range(B):
        if lens[b]:
            gl.append(b, kb[b, :, :lens[b]], vb[b, :, :lens[b]], 0)
    q = I.random_bf16(99, (B, 2, 128))
    out, lse = gl.decode(q)
    caches = [[O.build_head_cache(O.bf16_to_f32(kb[b, 0, :lens[b]]), O.bf16_to_f32(vb[b, 0, :lens[b]]), gl.spec)]
              for b in range(B)]
    out_ref, lse_ref = O.decode_attention(O.bf16_to_f32(q), caches)
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref)
    assert gl.status_value() == 0

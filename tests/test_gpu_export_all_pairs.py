"""Every (sequence, kv head) pair of full-size layers: the dequantized export, bit-exact.

The workload tests check attention on 6 to 16 sampled pairs per layer.  This
file checks what the cache holds for all of a layer's pairs, after the same
benchmark step (the cache of T - 1 tokens, then the step's append, folded into
the decode launch for FP8 layers without sink tokens): kvq_dequantize exports
each sequence's K and V in fp32, and the oracle rebuilds every pair from the
same seeded bf16 inputs.  Equal sha256 digests of the fp32 bit patterns mean
equal codes, scales, zero-points and bf16 parts, wherever they sit in the
block pool.  The oracle runs in spawned worker processes (numpy only); it gets
the inputs, never anything the CUDA path computed.

Covered, every pair: the paged mix's first INT8 and a middle INT4 layer (64
ragged sequences of 1K-64K tokens x 8 heads), the 70B INT4 layer, the INT2 32K
MHA layer (32 x 32 pairs; its step spills a Key group from the residual
window), the FP8 E4M3 and E5M2 layers (append folded into the decode), the FP8
layer with two query tokens, the bf16 skip layer, and the pre-RoPE and
dense-and-sparse INT4 layers.
"""
import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np
import pytest

from oracle import kvq_oracle as O
from quantized_kv_cache_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bench  # noqa: E402
import oracle_export as OE  # noqa: E402
from quantized_kv_cache_decode_gb300 import kvq  # noqa: E402

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def pool():
    workers = max(1, min(16, os.cpu_count() or 1))
    with cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn")) as ex:
        yield ex, workers


def _spec(fmt):
    fp8 = bench.is_fp8(fmt)
    return O.Spec(fmt.fmt, d=128, G=1 if fp8 else fmt.G, Gv=fmt.Gv, R=0 if fp8 else fmt.R, S=fmt.S,
                  rope_base=fmt.rope_base, k_outliers=fmt.k_outliers, v_outliers=fmt.v_outliers)


def _bits(t):
    # bf16 device tensor -> uint16 bit patterns on the host
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_all_pairs(pool, w, l, seqs=None):
    ex, workers = pool
    fmt = w.layer_formats[l]
    spec = _spec(fmt)
    n_app = max(1, w.append_tokens)
    uniform = w.seq_len_range is None
    lens_after = np.full(w.batch, w.seq_len) if uniform else I.seq_lens(w) + w.append_tokens
    lens_before = [int(t) - n_app for t in lens_after]
    lay = bench.Layer(kvq, torch, w, l, fmt, lens_before, n_app, DEV, seed_offset=0)
    lay.step_calls()
    torch.cuda.synchronize()
    assert lay.status.item() == 0
    H = w.num_kv_heads
    seqs = range(w.batch) if seqs is None else seqs
    ks = vs = None
    if uniform:
        kd, vd = I.device_kv_bf16(w, l, int(lens_after[0]), DEV, batch=w.batch)
        if spec.is_fp8:  # per-tensor scales over the whole layer, as the calibration computes them
            ks = O.fp8_tensor_scale(kd.float().cpu().numpy(), spec.fmt)
            vs = O.fp8_tensor_scale(vd.float().cpu().numpy(), spec.fmt)
            assert lay.cache.k_tensor_scale.item() == float(ks)
            assert lay.cache.v_tensor_scale.item() == float(vs)
    pending, bad, checked = [], [], 0

    def settle(limit):
        nonlocal checked
        while len(pending) > limit:
            (b, h), fut, kg, vg = pending.pop(0)
            kr, vr = fut.result()
            if (kr, vr) != (kg, vg):
                bad.append((b, h, "K" if kr != kg else "", "V" if vr != vg else ""))
            checked += 1

    for b in seqs:
        T = int(lens_after[b])
        if uniform:
            kb, vb = _bits(kd[b]), _bits(vd[b])
        else:
            wb = I.Workload(**{**w.__dict__, "batch": 1})
            k1, v1 = I.device_kv_bf16(wb, l, T, DEV, batch=1, seed_offset=7 * b)
            kb, vb = _bits(k1[0]), _bits(v1[0])
            del k1, v1
        ko = torch.empty((1, H, T, 128), dtype=torch.float32, device=DEV)
        vo = torch.empty_like(ko)
        kvq.dequantize(lay.cfg, lay.cache.seq_struct(b), lay.lens_after[b:b + 1], 1, T, ko, vo, lay.status)
        torch.cuda.synchronize()
        kh, vh = ko[0].cpu().numpy(), vo[0].cpu().numpy()
        del ko, vo
        for h in range(H):
            fut = ex.submit(OE.export_digests, spec, kb[h], vb[h], n_app, ks, vs)
            pending.append(((b, h), fut, OE.digest(kh[h]), OE.digest(vh[h])))
        settle(4 * workers)  # bound the inputs held for the workers
    settle(0)
    assert lay.status.item() == 0
    assert checked == len(list(seqs)) * H
    assert not bad, f"{len(bad)} of {checked} pairs differ from the oracle's export, e.g. {bad[:8]}"


@pytest.mark.parametrize("layer", [0, 31])
def test_paged_mixed_every_pair(pool, layer):
    _check_all_pairs(pool, I.WORKLOADS["paged_mixed_int8_int4_64l"](), layer)


def test_llama3_70b_int4_every_pair(pool):
    _check_all_pairs(pool, I.WORKLOADS["llama3_70b_kivi_int4_80l"](), 0)


@pytest.mark.parametrize("name", ["llama3_8b_fp8_e4m3", "llama3_8b_fp8_e5m2", "llama3_8b_fp8_e4m3_2q",
                                  "llama3_8b_bf16_skip_layer", "llama3_8b_kivi_int4_prerope",
                                  "llama3_8b_kivi_int4_sparse"])
def test_llama3_8b_every_pair(pool, name):
    _check_all_pairs(pool, I.WORKLOADS[name](), 0)


def test_llama2_7b_int2_spill_every_pair(pool):
    _check_all_pairs(pool, I.WORKLOADS["llama2_7b_kivi2_int2_32k"](), 0)

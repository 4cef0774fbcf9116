"""GPU parity of libkvq against the CPU oracle, through the C ABI.

Small shapes that still span several 16-token tiles, several CTAs and ragged
tails, over every format, both layouts, GQA ratios 1..8 and edge lengths.
  * codes, scales, zero-points, sink and residual window: bit-exact;
  * kvq_dequantize export: bit-exact;
  * attention: max|out - ref| <= 2e-3 * max|ref| (fp32 output),
    |lse - ref| <= 1e-4, bf16 output == round-to-nearest-even of the fp32 output.
"""
import math
import zlib

import numpy as np
import pytest

from oracle import kvq_oracle as O
from quantized_kv_cache_decode_gb300 import inputs as I

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kvq_testlib as TL  # noqa: E402


def make_inputs(seed, H, g, lens, outliers=4, scale=10.0):
    rng = np.random.default_rng(seed)
    chans = rng.choice(128, size=outliers, replace=False)
    mask = np.zeros(128, bool)
    mask[chans] = True
    kv = {}
    for b, T in enumerate(lens):
        for h in range(H):
            k = I.random_bf16(seed * 1000 + 2 * (b * H + h), (T, 128), outlier_mask=mask, outlier_scale=scale)
            v = I.random_bf16(seed * 1000 + 2 * (b * H + h) + 1, (T, 128))
            kv[b, h] = (k, v)
    q = I.random_bf16(seed * 7 + 3, (len(lens), H * g, 128))
    return kv, q


def build(fmt, H, g, lens, G, Gv, R, S, paged, seed, block_tokens=16, chunks=None, rope_base=0.0, k_outliers=0,
          v_outliers=0):
    gl = TL.GpuLayer(fmt, H, lens, G, Gv, R, S, paged=paged, block_tokens=block_tokens, seed=seed,
                     rope_base=rope_base, k_outliers=k_outliers, v_outliers=v_outliers)
    kv, q = make_inputs(seed, H, g, lens)
    ks = vs = None
    if gl.fp8:
        kall = np.concatenate([kv[k][0].reshape(-1) for k in kv] + [np.zeros(0, np.uint16)])
        vall = np.concatenate([kv[k][1].reshape(-1) for k in kv] + [np.zeros(0, np.uint16)])
        gl.calibrate_fp8(kall, vall)
        ks = O.fp8_tensor_scale(O.bf16_to_f32(kall), fmt)
        vs = O.fp8_tensor_scale(O.bf16_to_f32(vall), fmt)
        assert gl.layer.k_tensor_scale.item() == float(ks) and gl.layer.v_tensor_scale.item() == float(vs)
    for b, T in enumerate(lens):
        if T == 0:
            continue
        kb = np.stack([kv[b, h][0] for h in range(H)])
        vb = np.stack([kv[b, h][1] for h in range(H)])
        steps = chunks(T) if chunks else [T]
        t0 = 0
        for n in steps:
            gl.append(b, kb[:, t0:t0 + n], vb[:, t0:t0 + n], t0)
            t0 += n
        assert t0 == T
    torch.cuda.synchronize()
    caches = [[O.build_head_cache(O.bf16_to_f32(kv[b, h][0]), O.bf16_to_f32(kv[b, h][1]), gl.spec, ks, vs)
               for h in range(H)] for b in range(len(lens))]
    return gl, caches, q


CASES = [
    # fmt, H, g, lens, G, Gv, R, S, paged, block
    # one long sequence over every SM: each pair merges more than 64 partials
    ("fp8_e4m3", 1, 8, [40000], 1, 128, 0, 1, False, 16),
    ("int4", 1, 4, [30000], 32, 128, 32, 0, False, 16),
    ("int8", 1, 6, [25000], 16, 128, 64, 1, False, 16),  # 8-warp CTAs, one-tile records, many partials
    # 128 ragged pairs: the pair-aligned FP8 grid with pairs cut across CTAs
    ("fp8_e4m3", 8, 4, [16 + 37 * i for i in range(16)], 1, 128, 0, 0, False, 16),
    ("int4", 2, 4, [512], 32, 128, 32, 0, False, 16),
    ("int4", 2, 4, [0, 1, 31, 63, 64, 65, 700], 32, 128, 32, 0, False, 16),
    ("int2", 3, 1, [1000, 129, 160, 161, 5], 32, 32, 128, 0, False, 16),
    ("int8", 2, 6, [300, 17, 80, 81, 2], 16, 128, 64, 1, False, 16),
    ("int4", 2, 8, [777, 2000, 1], 128, 64, 128, 2, False, 16),
    ("int2", 1, 5, [600, 47], 16, 16, 0, 0, False, 16),
    ("fp8_e4m3", 2, 4, [0, 1, 15, 16, 17, 333], 1, 128, 0, 0, False, 16),
    ("fp8_e4m3", 2, 3, [100, 257, 3], 1, 128, 0, 1, False, 16),
    ("int4", 2, 6, [300, 1000, 17, 81], 16, 128, 64, 1, True, 16),
    ("int8", 3, 2, [250, 96, 97], 16, 32, 64, 1, True, 16),
    ("int2", 2, 2, [900, 33], 32, 16, 32, 0, True, 32),
    ("fp8_e4m3", 2, 4, [500, 7, 48], 1, 128, 0, 1, True, 16),
    ("fp8_e4m3", 1, 8, [400, 31], 1, 128, 0, 0, True, 32),
    ("fp8_e5m2", 2, 4, [0, 1, 15, 16, 17, 333], 1, 128, 0, 0, False, 16),
    ("fp8_e5m2", 2, 6, [500, 7, 48], 1, 128, 0, 1, True, 16),
    ("fp8_e5m2", 1, 8, [1200, 64], 1, 128, 0, 2, False, 16),
    ("bf16", 2, 4, [0, 1, 15, 16, 17, 333], 0, 0, 0, 0, False, 16),
    ("bf16", 2, 8, [700, 31, 2], 0, 0, 0, 1, False, 16),
    ("bf16", 1, 1, [1500, 160], 0, 0, 0, 3, False, 16),
    # the largest Key groups (256 tokens: 16 tiles per record, the spill's largest staging)
    ("int4", 1, 4, [1200, 300, 511, 512], 256, 128, 256, 0, False, 16),
    ("int8", 2, 8, [900, 767], 256, 64, 32, 1, False, 16),
    ("int2", 1, 2, [1300, 40], 256, 32, 0, 0, False, 16),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-H{c[1]}g{c[2]}-G{c[4]}Gv{c[5]}R{c[6]}S{c[7]}"
                                             f"{'-paged' if c[8] else ''}" for c in CASES])
def test_parity(case):
    fmt, H, g, lens, G, Gv, R, S, paged, blk = case
    seed = zlib.crc32(repr(case).encode()) % 10000  # stable across processes
    gl, caches, q = build(fmt, H, g, lens, G, Gv, R, S, paged, seed, block_tokens=blk)
    B = len(lens)
    # stored cache, bit-exact
    for b, T in enumerate(lens):
        for h in range(H):
            TL.compare_logical(gl.logical(b, h, T), caches[b][h])
    # dequantized export, bit-exact
    Tmax = max(lens) + 3
    ko, vo = gl.dequantize(Tmax)
    for b, T in enumerate(lens):
        for h in range(H):
            kr, vr = O.dequantized_f32(caches[b][h])
            assert np.array_equal(ko[b, h, :T].view(np.uint32), kr.view(np.uint32))
            assert np.array_equal(vo[b, h, :T].view(np.uint32), vr.view(np.uint32))
            assert np.all(ko[b, h, T:] == 0) and np.all(vo[b, h, T:] == 0)
    # attention
    qf = O.bf16_to_f32(q)
    out_ref, lse_ref = O.decode_attention(qf, caches)
    out, lse = gl.decode(q)
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref)
    out16, lse16 = gl.decode(q, out_bf16=True)
    assert torch.equal(out16, out.to(torch.bfloat16))
    assert torch.equal(lse16, lse)
    assert gl.status_value() == 0


MULTI = [
    # fmt, H, query heads per kv head, query tokens M, lens, G, Gv, R, S, paged
    ("int4", 2, 4, 2, [300, 1, 17, 64], 16, 128, 32, 1, False),
    ("fp8_e4m3", 2, 2, 4, [500, 3, 48, 1000], 1, 128, 0, 0, False),
    ("int8", 1, 1, 8, [250, 7, 129], 16, 64, 16, 0, True),
    ("bf16", 2, 4, 2, [333, 2], 0, 0, 0, 1, False),
    ("int2", 2, 3, 2, [200, 40], 32, 32, 64, 0, False),
    ("fp8_e5m2", 1, 1, 3, [70, 2], 1, 128, 0, 1, True),
]


@pytest.mark.parametrize("case", MULTI, ids=[f"{c[0]}-H{c[1]}g{c[2]}M{c[3]}{'-paged' if c[9] else ''}" for c in MULTI])
def test_multi_query_parity(case):
    # M query tokens per sequence (the cache's last M tokens), each attending causally
    fmt, H, gh, M, lens, G, Gv, R, S, paged = case
    seed = zlib.crc32(repr(case).encode()) % 10000  # stable across processes
    gl, caches, _ = build(fmt, H, gh, lens, G, Gv, R, S, paged, seed)
    q = I.random_bf16(seed * 3 + 1, (len(lens), M, H * gh, 128))
    out_ref, lse_ref = O.decode_attention_multi(O.bf16_to_f32(q), caches)
    out, lse = gl.decode_multi(q)
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref)
    out16, lse16 = gl.decode_multi(q, out_bf16=True)
    assert torch.equal(out16, out.to(torch.bfloat16)) and torch.equal(lse16, lse)
    # the last query token alone is the plain decode step, bit for bit
    o1, l1 = gl.decode(np.ascontiguousarray(q[:, -1]))
    o2, l2 = gl.decode_multi(np.ascontiguousarray(q[:, -1:]))
    assert torch.equal(o1, o2[:, 0]) and torch.equal(l1, l2[:, 0])
    assert gl.status_value() == 0


@pytest.mark.parametrize("fmt,G,Gv,R,S", [("int4", 32, 128, 32, 1), ("fp8_e4m3", 1, 128, 0, 0), ("bf16", 0, 0, 0, 1),
                                          ("int2", 16, 32, 16, 0)])
def test_sequence_split_lse_merge(fmt, G, Gv, R, S):
    # each sequence's tokens split in two parts held by separate caches (as two devices of a
    # sequence-parallel decode would hold them; part B has no sink); each part decoded with its
    # lse, the two merged by kvq_lse_merge == the oracle's attention over all the tokens
    from quantized_kv_cache_decode_gb300 import kvq
    H, g = 2, 4
    la, lb = [700, 33, 200], [301, 64, 0]
    B, Hq = len(la), H * g
    kv, q = make_inputs(31, H, g, [a + b for a, b in zip(la, lb)])
    parts = []
    for lens, s_sink, off, seed in ((la, S, 0, 3), (lb, 0, 1, 4)):
        gl = TL.GpuLayer(fmt, H, lens, G, Gv, R, s_sink, seed=seed)
        sl = [slice(0, la[b]) if off == 0 else slice(la[b], la[b] + lb[b]) for b in range(B)]
        ks = vs = None
        if gl.fp8:
            kall = np.concatenate([kv[b, h][0][sl[b]].reshape(-1) for b in range(B) for h in range(H)])
            vall = np.concatenate([kv[b, h][1][sl[b]].reshape(-1) for b in range(B) for h in range(H)])
            gl.calibrate_fp8(kall, vall)
            ks, vs = O.fp8_tensor_scale(O.bf16_to_f32(kall), fmt), O.fp8_tensor_scale(O.bf16_to_f32(vall), fmt)
        for b in range(B):
            if lens[b]:
                gl.append(b, np.stack([kv[b, h][0][sl[b]] for h in range(H)]),
                          np.stack([kv[b, h][1][sl[b]] for h in range(H)]), 0)
        torch.cuda.synchronize()
        caches = [[O.build_head_cache(O.bf16_to_f32(kv[b, h][0][sl[b]]), O.bf16_to_f32(kv[b, h][1][sl[b]]), gl.spec,
                                      ks, vs) for h in range(H)] for b in range(B)]
        o, l = gl.decode(q)
        assert gl.status_value() == 0
        parts.append((o, l, caches))
    o_parts = torch.stack([parts[0][0], parts[1][0]]).contiguous()
    l_parts = torch.stack([parts[0][1], parts[1][1]]).contiguous()
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    kvq.lse_merge(o_parts, l_parts, 2, B * Hq, out, False, lse)
    out16 = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    kvq.lse_merge(o_parts, l_parts, 2, B * Hq, out16, True)
    torch.cuda.synchronize()
    qf = O.bf16_to_f32(q)
    ref_o = np.zeros((B, Hq, 128))
    ref_l = np.zeros((B, Hq))
    for b in range(B):
        for h in range(H):
            ka, va = O.dequantized_f64(parts[0][2][b][h])
            kb, vb = O.dequantized_f64(parts[1][2][b][h])
            kh, vh = np.concatenate([ka, kb]), np.concatenate([va, vb])
            for j in range(g):
                ref_o[b, h * g + j], ref_l[b, h * g + j] = O.attend_head(qf[b, h * g + j], kh, vh, 1 / math.sqrt(128))
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
    assert torch.equal(out16, out.to(torch.bfloat16))


@pytest.mark.parametrize("fmt,G,Gv,R,S", [("int4", 32, 128, 32, 0), ("int2", 32, 32, 64, 1),
                                          ("int8", 16, 64, 16, 2), ("fp8_e4m3", 1, 128, 0, 1),
                                          ("fp8_e5m2", 1, 128, 0, 0), ("bf16", 0, 0, 0, 1)])
def test_incremental_appends_equal_bulk(fmt, G, Gv, R, S):
    lens = [203, 77]

    def chunks(T):
        out, t, i = [], 0, 0
        pattern = [1, 1, 5, 1, 40, 1, 1, 33, 2]
        while t < T:
            n = min(pattern[i % len(pattern)], T - t)
            out.append(n)
            t += n
            i += 1
        return out

    gl, caches, q = build(fmt, 2, 3, lens, G, Gv, R, S, False, 123, chunks=chunks)
    for b, T in enumerate(lens):
        for h in range(2):
            TL.compare_logical(gl.logical(b, h, T), caches[b][h])
    out, lse = gl.decode(q)
    out_ref, lse_ref = O.decode_attention(O.bf16_to_f32(q), caches)
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref)
    assert gl.status_value() == 0


@pytest.mark.parametrize("fmt", ["int4", "fp8_e4m3"])
def test_paged_equals_contiguous_and_permutation_invariant(fmt):
    lens = [700, 129, 64]
    G = 1 if fmt == "fp8_e4m3" else 16
    gc, _, q = build(fmt, 2, 4, lens, G, 128, 32 if G > 1 else 0, 1, False, 5)
    gp, _, _ = build(fmt, 2, 4, lens, G, 128, 32 if G > 1 else 0, 1, True, 5)
    oc, lc = gc.decode(q)
    op, lp = gp.decode(q)
    assert torch.equal(oc, op) and torch.equal(lc, lp)
    gp2, _, _ = build(fmt, 2, 4, lens, G, 128, 32 if G > 1 else 0, 1, True, 6)  # other block permutation
    assert not np.array_equal(gp2.table_np, gp.table_np)
    # same data, different table: outputs identical bit for bit
    gp3, _, _ = build(fmt, 2, 4, lens, G, 128, 32 if G > 1 else 0, 1, True, 5)
    o3, l3 = gp3.decode(q)
    assert torch.equal(o3, op) and torch.equal(l3, lp)


def test_bad_block_and_capacity_are_reported_not_faulted():
    from quantized_kv_cache_decode_gb300 import kvq
    lens = [300, 200]
    gl, caches, q = build("int4", 2, 4, lens, 16, 128, 32, 0, True, 9)
    # corrupt one block-table entry (host-made fault): the kernel must skip that tile and report
    bad = gl.table_np.copy()
    bad[0, 3] = gl.cfg.num_blocks + 5
    gl.layer.block_table.copy_(torch.from_numpy(bad))
    gl.status.zero_()
    out, lse = gl.decode(q)
    assert gl.status_value() & kvq.DEV_BAD_BLOCK
    assert torch.isfinite(out).all()
    # a length beyond the capacity: reported and clamped
    gl.layer.block_table.copy_(torch.from_numpy(gl.table_np))
    gl.status.zero_()
    out, lse = gl.decode(q, lens=[300, 10 ** 6])
    assert gl.status_value() & kvq.DEV_CAPACITY
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "int4"])
def test_append_decode_past_capacity_is_reported_not_stored(fmt):
    # a full store: the step's token cannot be stored; the call reports
    # KVQ_DEV_CAPACITY, writes nothing, and attends over the tokens the store holds
    from quantized_kv_cache_decode_gb300 import kvq
    G = 1 if fmt == "fp8_e4m3" else 16
    lens = [32, 32] if fmt == "fp8_e4m3" else [47, 47]  # the most each store holds (INT4: 32 + a 15-token window)
    gl, caches, q = build(fmt, 2, 4, lens, G, 128, 0, 0, False, 31)
    names = ("qstore",) if fmt == "fp8_e4m3" else ("qstore", "resid_k", "resid_v")
    before = {name: gl.raw(name).copy() for name in names}
    kb = I.random_bf16(77, (len(lens), 2, 128))
    vb = I.random_bf16(78, (len(lens), 2, 128))
    gl.status.zero_()
    out, lse = gl.append_decode(kb, vb, q, lens)
    assert gl.status_value() & kvq.DEV_CAPACITY
    for name, raw in before.items():
        assert np.array_equal(gl.raw(name), raw)
    out_ref, lse_ref = O.decode_attention(O.bf16_to_f32(q), caches)
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref)


def test_bounded_wait_runs_out_reports_and_context_stays_usable():
    # self-test hook: one warp's first copy is withheld while its barrier expects the bytes,
    # so its bounded wait (about a second) gives up; the launch reports KVQ_DEV_TIMEOUT and
    # finishes, and the next call on the same context gives the oracle's result
    import time
    from quantized_kv_cache_decode_gb300 import kvq
    gl, caches, q = build("fp8_e4m3", 2, 4, [300, 40], 1, 128, 0, 0, False, 41)
    B, Hq = 2, 8
    qd = torch.from_numpy(q.astype(np.int16)).cuda()
    wsb = kvq.decode_workspace_size(gl.cfg, B, Hq)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    gl.status.zero_()
    t0 = time.time()
    kvq.selftest_bounded_wait(gl.cfg, gl.layer.struct(), qd, Hq, gl.seq_lens_dev(), B, 1 / math.sqrt(128), out, False,
                              lse, ws, wsb, gl.status)
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert gl.status_value() & kvq.DEV_TIMEOUT
    assert 0.3 < waited < 30.0, waited
    gl.status.zero_()
    o, l = gl.decode(q)
    TL.check_attention(o.cpu().numpy(), l.cpu().numpy(), *O.decode_attention(O.bf16_to_f32(q), caches))
    assert gl.status_value() == 0


def test_workspace_too_small_is_rejected():
    from quantized_kv_cache_decode_gb300 import kvq
    gl, _, q = build("int4", 1, 2, [64], 16, 128, 16, 0, False, 3)
    wsb = kvq.decode_workspace_size(gl.cfg, 1, 2)
    ws = torch.empty(wsb - 16, dtype=torch.uint8, device="cuda")
    out = torch.empty((1, 2, 128), dtype=torch.float32, device="cuda")
    sl = torch.tensor([64], dtype=torch.int32, device="cuda")
    qd = torch.from_numpy(q.astype(np.int16)).cuda()
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attention(gl.cfg, gl.layer.struct(), qd, 2, sl, 1, 0.1, out, False, None, ws, wsb - 16)
    assert e.value.status == -4


@pytest.mark.parametrize("fmt,lens", [("int4", [2000, 700, 33]), ("fp8_e4m3", [4000, 17, 900]),
                                      # equal lengths: whole pairs per CTA (128 pairs: one each; 256: two each)
                                      ("int4", [300] * 64), ("int4", [100] * 128), ("fp8_e4m3", [200] * 64)],
                         ids=["int4-ragged", "fp8-ragged", "int4-128pairs", "int4-256pairs", "fp8-128pairs"])
def test_fused_combine_equals_two_launches_and_repeats(fmt, lens):
    # kvq_decode_attention merges partials inside the decode launch (arrival counters in the
    # workspace); kvq_decode_partials + kvq_decode_combine do it in two launches.  Same bits,
    # and the counters are back at zero after every call.
    from quantized_kv_cache_decode_gb300 import kvq
    G = 1 if fmt == "fp8_e4m3" else 32
    gl, caches, q = build(fmt, 2, 4, lens, G, 128, 32 if G > 1 else 0, 0, False, 21)
    o1, l1 = gl.decode(q)
    B, Hq = len(lens), 8
    TL.check_attention(o1.cpu().numpy(), l1.cpu().numpy(), *O.decode_attention(O.bf16_to_f32(q), caches))
    qd = torch.from_numpy(q.astype(np.int16)).cuda()
    wsb = kvq.decode_workspace_size(gl.cfg, B, Hq)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    sl = gl.seq_lens_dev()
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    for _ in range(3):
        kvq.decode_attention(gl.cfg, gl.layer.struct(), qd, Hq, sl, B, 1 / math.sqrt(128), out, False, lse, ws, wsb)
        torch.cuda.synchronize()
        assert torch.equal(out, o1) and torch.equal(lse, l1)
    cnt = ws[-B * 2 * 4:].view(torch.int32)
    assert int(cnt.abs().sum()) == 0
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    kvq.decode_partials(gl.cfg, gl.layer.struct(), qd, Hq, sl, B, 1 / math.sqrt(128), ws, wsb)
    kvq.decode_combine(gl.cfg, Hq, B, out2, False, lse2, ws, wsb)
    torch.cuda.synchronize()
    assert torch.equal(out2, o1) and torch.equal(lse2, l1)


ROPE_CASES = [
    # fmt, H, g, lens, G, Gv, R, S, paged, block, rope_base: Keys appended before RoPE, rotated at
    # their positions by the decode ("KV Cache Quantization Analysis", section 3 RoPE bullet)
    ("int4", 2, 4, [700, 33, 129, 0], 32, 128, 32, 1, False, 16, 10000.0),
    ("int8", 2, 6, [300, 17, 80, 81, 2], 16, 128, 64, 1, True, 16, 500000.0),
    ("int2", 3, 1, [1000, 160, 5], 32, 64, 128, 0, False, 16, 10000.0),
    ("int4", 2, 8, [500, 96], 16, 64, 16, 2, True, 16, 500000.0),
    # long positions (angles up to 20000 turns of the fastest pair), several CTAs per pair
    ("int4", 1, 8, [20000], 128, 128, 128, 2, False, 16, 500000.0),
]


@pytest.mark.parametrize("case", ROPE_CASES, ids=[f"{c[0]}-H{c[1]}g{c[2]}-G{c[4]}Gv{c[5]}R{c[6]}S{c[7]}"
                                                  f"{'-paged' if c[8] else ''}-base{int(c[10])}" for c in ROPE_CASES])
def test_pre_rope_parity(case):
    fmt, H, g, lens, G, Gv, R, S, paged, blk, base = case
    seed = zlib.crc32(repr(case).encode()) % 10000
    gl, caches, q = build(fmt, H, g, lens, G, Gv, R, S, paged, seed, block_tokens=blk, rope_base=base)
    # the stored cache holds the Keys as appended (before the rotation), bit-exact
    for b, T in enumerate(lens):
        for h in range(H):
            TL.compare_logical(gl.logical(b, h, T), caches[b][h])
    ko, vo = gl.dequantize(max(lens) + 1)
    for b, T in enumerate(lens):
        for h in range(H):
            kr, vr = O.dequantized_f32(caches[b][h])
            assert np.array_equal(ko[b, h, :T].view(np.uint32), kr.view(np.uint32))
    # attention over the Keys rotated at their positions
    out_ref, lse_ref = O.decode_attention(O.bf16_to_f32(q), caches)
    out, lse = gl.decode(q)
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref)
    out16, lse16 = gl.decode(q, out_bf16=True)
    assert torch.equal(out16, out.to(torch.bfloat16)) and torch.equal(lse16, lse)
    assert gl.status_value() == 0


OUTLIER_CASES = [
    # fmt, H, g, lens, G, Gv, R, S, paged, k_outliers, v_outliers: dense-and-sparse rows
    # ("KV Cache Quantization Analysis", section 4, KVQuant item (iv))
    ("int4", 2, 4, [700, 33, 129, 0], 32, 128, 32, 1, False, 2, 2),
    ("int2", 2, 6, [300, 17, 80, 81, 2], 16, 64, 64, 1, True, 1, 3),
    ("int8", 3, 1, [1000, 160, 5], 32, 128, 128, 0, False, 8, 0),
    ("int4", 2, 8, [500, 96], 16, 128, 16, 2, True, 0, 8),
    ("int4", 1, 8, [20000], 128, 64, 128, 2, False, 3, 1),
]


@pytest.mark.parametrize("case", OUTLIER_CASES, ids=[f"{c[0]}-H{c[1]}g{c[2]}-G{c[4]}Gv{c[5]}R{c[6]}S{c[7]}"
                                                     f"{'-paged' if c[8] else ''}-k{c[9]}v{c[10]}" for c in OUTLIER_CASES])
def test_dense_and_sparse_parity(case):
    fmt, H, g, lens, G, Gv, R, S, paged, nk, nv = case
    seed = zlib.crc32(repr(case).encode()) % 10000
    gl, caches, q = build(fmt, H, g, lens, G, Gv, R, S, paged, seed, k_outliers=nk, v_outliers=nv)
    # codes of the dense part, scales, zero-points and the sparse lists: bit-exact
    for b, T in enumerate(lens):
        for h in range(H):
            TL.compare_logical(gl.logical(b, h, T), caches[b][h])
    ko, vo = gl.dequantize(max(lens) + 1)
    for b, T in enumerate(lens):
        for h in range(H):
            kr, vr = O.dequantized_f32(caches[b][h])
            assert np.array_equal(ko[b, h, :T].view(np.uint32), kr.view(np.uint32))
            assert np.array_equal(vo[b, h, :T].view(np.uint32), vr.view(np.uint32))
    out_ref, lse_ref = O.decode_attention(O.bf16_to_f32(q), caches)
    out, lse = gl.decode(q)
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref)
    out16, lse16 = gl.decode(q, out_bf16=True)
    assert torch.equal(out16, out.to(torch.bfloat16)) and torch.equal(lse16, lse)
    assert gl.status_value() == 0


APPEND_DECODE = [
    # fmt, H, g, lens after the step, G, Gv, R, S, paged, block
    # FP8 without sink tokens: the append folded into the decode launch; tokens that start a
    # tile (T = 1, 17, 33) and tokens inside one
    ("fp8_e4m3", 2, 4, [1, 16, 17, 20, 33, 300], 1, 128, 0, 0, False, 16),
    ("fp8_e5m2", 2, 4, [1, 17, 48, 129], 1, 128, 0, 0, True, 16),
    ("fp8_e4m3", 1, 8, [33, 400], 1, 128, 0, 0, True, 32),
    ("fp8_e4m3", 8, 4, [16 + 37 * i for i in range(16)], 1, 128, 0, 0, False, 16),
    ("fp8_e4m3", 1, 4, [20001], 1, 128, 0, 0, False, 16),
    # the other layers: the append launch(es), then the decode
    ("fp8_e4m3", 2, 4, [1, 2, 300], 1, 128, 0, 1, False, 16),
    ("int4", 2, 4, [1, 64, 65, 96, 700], 32, 128, 32, 0, False, 16),
    ("int2", 3, 1, [161, 5], 32, 32, 128, 0, False, 16),
    ("int8", 2, 6, [81, 2, 144], 16, 128, 64, 1, True, 16),
    ("bf16", 2, 4, [1, 333], 0, 0, 0, 1, False, 16),
]


@pytest.mark.parametrize("case", APPEND_DECODE, ids=[f"{c[0]}-H{c[1]}g{c[2]}-S{c[7]}{'-paged' if c[8] else ''}-"
                                                    f"{len(c[3])}seq" for c in APPEND_DECODE])
def test_append_decode_step(case):
    """kvq_append_decode_attention: the cache holds T - 1 tokens, the call appends token T - 1 and
    attends over all T.  The stored cache equals the oracle's over all T tokens (bit-exact), the
    attention equals the oracle's, and a plain decode over the result gives the same bits."""
    fmt, H, g, lens, G, Gv, R, S, paged, blk = case
    seed = zlib.crc32(repr(case).encode()) % 10000
    gl = TL.GpuLayer(fmt, H, lens, G, Gv, R, S, paged=paged, block_tokens=blk, seed=seed)
    kv, q = make_inputs(seed, H, g, lens)
    ks = vs = None
    if gl.fp8:  # the per-tensor scales from every token of the layer, the step's included
        kall = np.concatenate([kv[k][0].reshape(-1) for k in kv])
        vall = np.concatenate([kv[k][1].reshape(-1) for k in kv])
        gl.calibrate_fp8(kall, vall)
        ks = O.fp8_tensor_scale(O.bf16_to_f32(kall), fmt)
        vs = O.fp8_tensor_scale(O.bf16_to_f32(vall), fmt)
    for b, T in enumerate(lens):
        if T > 1:
            gl.append(b, np.stack([kv[b, h][0][:T - 1] for h in range(H)]),
                      np.stack([kv[b, h][1][:T - 1] for h in range(H)]), 0)
    torch.cuda.synchronize()
    knew = np.stack([np.stack([kv[b, h][0][T - 1] for h in range(H)]) for b, T in enumerate(lens)])
    vnew = np.stack([np.stack([kv[b, h][1][T - 1] for h in range(H)]) for b, T in enumerate(lens)])
    out, lse = gl.append_decode(knew, vnew, q, [T - 1 for T in lens])
    assert gl.status_value() == 0
    caches = [[O.build_head_cache(O.bf16_to_f32(kv[b, h][0]), O.bf16_to_f32(kv[b, h][1]), gl.spec, ks, vs)
               for h in range(H)] for b in range(len(lens))]
    for b, T in enumerate(lens):
        for h in range(H):
            TL.compare_logical(gl.logical(b, h, T), caches[b][h])
    out_ref, lse_ref = O.decode_attention(O.bf16_to_f32(q), caches)
    TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref)
    out2, lse2 = gl.decode(q)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)

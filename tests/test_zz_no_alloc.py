"""The allocation-free decode entry point (kvq_decode_attention_static_scratch).

Some callers cannot allocate device memory (their host application owns all of
it through its own pool, or an allocation's synchronisation is not allowed in
their loop).  This entry point uses a fixed scratch array inside the library
instead of a caller workspace.  The test calls it through the C ABI on two
different problems in a row -- one long sequence spread over many CTAs (many
partials in the shared array), then a short ragged batch with another query and
another split -- and checks each result against kvq_decode_attention (which
takes a workspace), within the attention tolerance used everywhere in the tests.
If the second call read partials or prefixes the first one left behind in the
shared array, its result would differ.

This file is collected last on purpose; it builds its own small caches, so it
passes alone in a fresh process as well as after the other tests.
"""
import ctypes
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kvq_testlib as TL  # noqa: E402
from quantized_kv_cache_decode_gb300 import inputs as I  # noqa: E402


def _layer(H, lens, seed):
    gl = TL.GpuLayer("int4", H, lens, 32, 128, 32, 1, seed=seed)
    for b, T in enumerate(lens):
        k = np.stack([I.random_bf16(seed * 1000 + 100 * b + h, (T, 128)) for h in range(H)])
        v = np.stack([I.random_bf16(seed * 1000 + 100 * b + h + 50, (T, 128)) for h in range(H)])
        gl.append(b, k, v, 0)
    return gl


def _static_scratch(gl, q, H, g, out_bf16=0, out=None):
    from quantized_kv_cache_decode_gb300 import kvq
    B = len(gl.lens)
    qd = torch.from_numpy(q.astype(np.int16)).cuda()
    if out is None:
        out = torch.full((B, H * g, 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, H * g), float("nan"), dtype=torch.float32, device="cuda")
    sl = gl.seq_lens_dev()
    st = kvq._lib.kvq_decode_attention_static_scratch(
        ctypes.byref(gl.cfg), ctypes.byref(gl.layer.struct()), qd.data_ptr(), H * g, sl.data_ptr(), B,
        ctypes.c_float(1 / math.sqrt(128)), out.data_ptr(), out_bf16, lse.data_ptr(), gl.status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, out, lse


def test_static_scratch_matches_workspace_entry_point_on_two_different_calls():
    from quantized_kv_cache_decode_gb300 import kvq
    # call 1: one long sequence over every SM (its partials fill much of the array)
    H1, g1, lens1 = 1, 8, [30000]
    gl1 = _layer(H1, lens1, seed=8)
    q1 = I.random_bf16(5, (len(lens1), H1 * g1, 128))
    # call 2: a short ragged batch, other heads, other query, other split
    H2, g2, lens2 = 2, 4, [900, 33, 257, 0]
    gl2 = _layer(H2, lens2, seed=9)
    q2 = I.random_bf16(6, (len(lens2), H2 * g2, 128))
    refs = []
    for gl, q in ((gl1, q1), (gl2, q2)):
        o, l = gl.decode(q)  # kvq_decode_attention with a caller workspace
        refs.append((o.cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64)))
    for (gl, q, H, g), (ro, rl) in zip(((gl1, q1, H1, g1), (gl2, q2, H2, g2)), refs):
        st, out, lse = _static_scratch(gl, q, H, g)
        assert st == 0, kvq.status_string(st)
        TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), ro, rl)
        assert gl.status_value() == 0


def test_static_scratch_bad_arguments_enqueue_nothing():
    from quantized_kv_cache_decode_gb300 import kvq
    H, g, lens = 2, 4, [300, 40]
    gl = _layer(H, lens, seed=10)
    q = I.random_bf16(7, (len(lens), H * g, 128))
    sentinel = torch.full((len(lens), H * g, 128), 3.0, dtype=torch.float32, device="cuda")
    st, out, lse = _static_scratch(gl, q, H, g, out_bf16=2, out=sentinel)
    assert st == -1, kvq.status_string(st)
    assert torch.all(out == 3.0) and torch.all(torch.isnan(lse))


def test_static_scratch_rejects_too_large_problems():
    from quantized_kv_cache_decode_gb300 import kvq
    cfg = kvq.make_config("int4", 8, 16, 128, 16, 0, capacity_tokens=16)
    layer = kvq.CacheLayer(cfg, 2048)
    need = kvq.decode_workspace_size(cfg, 2048, 64)
    assert need > 8 << 20
    qd = torch.zeros((2048, 64, 128), dtype=torch.bfloat16, device="cuda")
    sl = torch.zeros(2048, dtype=torch.int32, device="cuda")
    out = torch.zeros((2048, 64, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attention_static_scratch(cfg, layer.struct(), qd, 64, sl, 2048, 0.1, out, False, None)
    assert e.value.status == -4

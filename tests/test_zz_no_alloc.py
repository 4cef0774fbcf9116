"""The allocation-free decode entry point (kvq_decode_attention_static_scratch).

Some callers cannot allocate device memory (their host application owns all of
it through its own pool, or an allocation's synchronisation is not allowed in
their loop).  This entry point uses a fixed scratch array inside the library
instead of a caller workspace.  The test calls it through the C ABI twice in a
row and checks each result against kvq_decode_attention (which takes a
workspace), within the attention tolerance used everywhere in the tests.

This file is collected last on purpose; it builds its own small cache, so it
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


def test_static_scratch_matches_workspace_entry_point_twice():
    from quantized_kv_cache_decode_gb300 import kvq
    H, g, lens = 2, 4, [900, 33, 257]
    gl = TL.GpuLayer("int4", H, lens, 32, 128, 32, 1, seed=8)
    rng = np.random.default_rng(8)
    for b, T in enumerate(lens):
        k = np.stack([I.random_bf16(100 * b + h, (T, 128)) for h in range(H)])
        v = np.stack([I.random_bf16(100 * b + h + 50, (T, 128)) for h in range(H)])
        gl.append(b, k, v, 0)
    q = I.random_bf16(5, (len(lens), H * g, 128))
    ref_out, ref_lse = gl.decode(q)  # kvq_decode_attention with a caller workspace
    ref_out, ref_lse = ref_out.cpu().numpy(), ref_lse.cpu().numpy()
    qd = torch.from_numpy(q.astype(np.int16)).cuda()
    sl = gl.seq_lens_dev()
    for _ in range(2):
        out = torch.full((len(lens), H * g, 128), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((len(lens), H * g), float("nan"), dtype=torch.float32, device="cuda")
        # through the C ABI directly
        st = kvq._lib.kvq_decode_attention_static_scratch(
            ctypes.byref(gl.cfg), ctypes.byref(gl.layer.struct()), qd.data_ptr(), H * g, sl.data_ptr(), len(lens),
            ctypes.c_float(1 / math.sqrt(128)), out.data_ptr(), 0, lse.data_ptr(), gl.status.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert st == 0, kvq.status_string(st)
        torch.cuda.synchronize()
        TL.check_attention(out.cpu().numpy(), lse.cpu().numpy(), ref_out.astype(np.float64),
                           ref_lse.astype(np.float64))
    assert gl.status_value() == 0


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

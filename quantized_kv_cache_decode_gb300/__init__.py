"""GB300-native (sm_103a) attention decode over a quantized KV cache.

``kvq``    -- ctypes binding of libkvq.so (the C ABI in include/kvq.h); importing
              it fails loudly when the library has not been built.
``inputs`` -- seeded synthetic workloads (shapes, bf16 draws), no method arithmetic.
``build``  -- compiles libkvq.so in-tree with nvcc for sm_103a.
"""


def build(force: bool = False) -> str:
    from .builder import build as _build
    return _build(force=force)

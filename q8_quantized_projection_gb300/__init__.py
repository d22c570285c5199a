"""Q8_0 quantized projection on one GB300 (sm_103a).

The computation lives in ``libq8proj.so`` (CUDA kernels behind the C ABI of
``include/q8proj.h``); ``native`` is its thin ctypes binding, ``build``
compiles it in tree, and ``synth`` draws the seeded synthetic inputs.
"""
__all__ = ["native", "build", "synth"]

"""CPU oracle for the Q8_0 quantized projection (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package; the CUDA library and its binding never do.
"""

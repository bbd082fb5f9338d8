"""GB300 (sm_103a) library for decode attention over QEvict's three-tier KV cache.

The compute path lives in ``csrc/`` (CUDA kernels behind a C ABI declared in
``include/qevict.h``); ``binding`` is a thin ctypes layer over that ABI and
``synth`` draws the seeded synthetic workloads.
"""

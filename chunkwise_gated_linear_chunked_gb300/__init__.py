"""GB300-native chunkwise gated linear attention (GLA) forward.

The compute path lives in ``csrc/`` (sm_103a CUDA kernels behind a C ABI, ``libgla.so``, declared in
``include/gla.h``); ``binding`` is a thin ctypes layer over that ABI (import it explicitly; it requires the
built library); ``inputs`` draws the seeded synthetic workloads; ``build`` compiles the library in-tree.
"""

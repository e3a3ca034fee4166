"""GB300-native chunkwise gated linear attention (GLA) forward.

The compute path lives in ``csrc/`` (sm_103a CUDA kernels behind a C ABI, ``libgla.so``); ``binding`` is a
thin ctypes layer over that ABI; ``inputs`` draws the seeded synthetic workloads.  The binding is imported
lazily so that ``inputs`` can be used without the compiled library.
"""

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name == "binding":
        from . import binding
        return binding
    if name == "inputs":
        from . import inputs
        return inputs
    raise AttributeError(name)

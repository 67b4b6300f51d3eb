"""GB300-native fused GQA decode attention (sm_103a).

The compute lives in ``libgqa_decode.so`` (CUDA kernels behind a C ABI declared in
``include/gqa_decode.h``).  ``binding`` is the thin ctypes layer over that ABI; ``build``
compiles it; ``workloads`` draws seeded synthetic inputs.  Importing this package loads
nothing: ``binding.load()`` loads the library and raises if it is missing.
"""
__all__ = ["binding", "build", "workloads"]

"""GB300-native paged KV cache: the hot path of a vLLM-style engine step.

The compute lives in ``libpagedkv.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/pagedkv.h``); ``binding`` is the thin ctypes layer
above it. ``synth`` builds seeded synthetic steps. Nothing here is imported
eagerly, so the generator works on machines without the library.
"""

__all__ = ["binding", "synth", "build"]

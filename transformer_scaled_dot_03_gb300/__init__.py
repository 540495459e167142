"""GB300-native (sm_103a) multi-head scaled dot-product attention forward.

``attn`` is the Python binding of the C-ABI library ``libattn_sm103a.so`` (built
by ``build.py``); ``inputs`` holds the seeded synthetic input generators.
The binding is imported lazily so that CPU-only users of ``inputs`` do not
need the CUDA library.
"""

__all__ = ["attn", "inputs", "build"]

"""GB300-native paged KV cache and PagedAttention decode.

The compute path lives in the CUDA library ``_build/libpa.so`` (sources in
``csrc/``) behind the C ABI declared in ``include/pa.h``; ``binding`` is the
thin ctypes layer over it with the same names.  ``synth`` draws seeded
synthetic inputs.
"""
